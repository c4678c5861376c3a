// Widening tensor-core split-KV partial kernel for sm_103a (tcgen05 kind::f16): int8 or FP8
// e4m3 KV with per-token fp32 K and V scales (head_dim 64, 128 or 256), or f16 / bf16 KV (head_dim
// 64 or 128); bf16 or f16 Q; up to 128 packed rows per KV head (GQA groups x query rows: the
// speculative-verify shape); block size 8..128.
//
// Every int8 and every e4m3 value is exact in f16, so the cache is widened to f16 in shared
// memory (int8: a byte permute and one packed subtraction per two values; e4m3: one packed
// conversion per two values) and both contractions run on the 16-bit tensor cores in f16; the
// scales stay outside them (the K scale multiplies the score column, the V scale the
// probability column). An f16 cache is copied as it is. A bf16 K tile enters f16 scaled by a
// power of two chosen from its largest value, which then stands as the tile's per-token scale;
// a bf16 V tile stays bf16, and the PV contraction runs in bf16 with P sent as a high part
// plus the bf16 rounding of its remainder (about 16 significant bits of P), so V keeps bf16's
// whole range. A bf16 Q row enters as f16 after a power-of-two scale that is undone on the
// scores.
//
// Persistent CTAs, one per SM, take the real (request, kv head, split) items of a work list
// built on the device from the lengths, in turn (item k to CTA k mod grid); per item each KV
// page of the split is read from HBM once (GQA packing: "split packed-Q8 verifier KV scans",
// hipfire PR #760, Summary). Roles (512 threads):
//   warp 0, 2     producers: walk the block table one tile ahead and TMA-load each page's K
//                 rows (warp 0) and V rows (warp 2), as stored, in 64-token tiles into staging
//                 rings of their own (K: 2 stages, V: 3), with the tile's scales (cp.async,
//                 quantised caches) and page mask;
//   warps 12..15  converters: widen staged tiles to f16 in the 128-byte-swizzle layout the
//                 MMAs read (rows = tokens, 64-element atoms), all four warps on each, in the
//                 order K(0), K(1), V(0), K(2), V(1), ...: K(j) into f16 K buffer j % 2 once the
//                 QK^T of tile j - 2 is done, V(j) into the f16 V buffer once the PV of tile
//                 j - 1 is done; the tile's scales, page mask and largest V scale go to a
//                 4-slot meta ring with K(j);
//   warp 1        one thread issues every QK^T: A = Q in TMEM (written once per item), B = the
//                 f16 K buffer (K-major), D = S in TMEM (two 64-column buffers);
//   warp 3        one thread issues every PV: A = P in shared memory (K-major, two buffers),
//                 B = the f16 V tile (MN-major, atoms 64 tokens x 128 B apart), D = O in TMEM;
//   warps 4..11   softmax: two threads per packed row (TMEM lane), one per 32-token half of
//                 the tile; they exchange their row maxima through shared memory, keep the same
//                 running (maximum, P scale) and their own partial sums. Online softmax in log2
//                 units (tiny-llm PR #11: per-split online (m, l, acc)); a row's exponent
//                 reference moves only when a tile's maximum passes it by more than kSlack, so O
//                 is rarely rescaled. P times the V scale is rounded once to f16 (2^-11
//                 relative; bf16 V: the high and low bf16 parts), with a power-of-two factor
//                 2^C that keeps it inside the 16-bit range: C follows the largest V scale
//                 seen, only ever decreases, and O is then rescaled exactly (each thread of a
//                 row its half of the columns).
//
// Every wait is bounded in time; a timeout sets TLLM_FLAG_TIMEOUT, lets every role run to its
// end without waiting, skips the output stores, takes no further item and frees TMEM.
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace tllm {
namespace {

using namespace ptx;

constexpr int kT = 64;                 // tokens per tile
constexpr int kThreads = 512;
constexpr uint32_t kFull = 0xffffffffu;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0, kColS = 128, kColO = 256;   // Q: D/2 columns, S: 2 x 64, O: D
constexpr int kEpiStride = 36;          // floats per staged output row (32 + 4: conflict-free float4 rows)
constexpr int kSmThreads = 256;         // softmax: 8 warps, two threads per TMEM lane
// Slack of a row's exponent reference M (log2 units): M moves only when a tile's row maximum
// passes it by more than kSlack, so P = 2^(score - M) stays below 2^kSlack and the O rescale (a
// TMEM round trip that waits for the previous tile's PV) is rare; the P scale 2^C leaves room.
constexpr int kSlack = 4;

__host__ __device__ constexpr uint32_t align1k(uint32_t x) { return (x + 1023u) & ~1023u; }

// Cache element types the kernel widens: int8 and e4m3 (exact in f16, per-token scales), f16
// (copied) and bf16 (scaled into f16 by a power of two per tile).
constexpr int kKvI8 = 0, kKvE4m3 = 1, kKvF16 = 2, kKvBf16 = 3;

template <int D, int kEsz, int kPParts>
struct Lay {
  static constexpr uint32_t kAtom = kT * 128;                 // bytes of one atom column of a tile
  static constexpr uint32_t kScT = kT * 4;                    // one operand's per-token scales
  static constexpr uint32_t kSc = 2 * kScT;                   // K scales | V scales
  static constexpr uint32_t kMeta = kSc + 16;                 // scales | page mask | largest V scale x2
  static constexpr uint32_t kRaw = kT * D * kEsz;             // one staged operand tile (K or V) as stored
  static constexpr uint32_t kStage = align1k(kRaw + kScT + 16);        // rows | scales | page mask, as stored
  // A 16-bit tile of head_dim 256 is 32 KB: that instance stages K and V one tile deep (the
  // converters then wait for a staged V tile when they widen it, not before its K tile) and,
  // for bf16 (two P parts), keeps one f16 K buffer, so that the stages fit the shared memory.
  static constexpr bool kBig16 = D == 256 && kEsz == 2;
  static constexpr int kStK = kBig16 ? 1 : 2, kStV = kBig16 ? 1 : 3;   // staging ring depths: K, V
  static constexpr int kNK16 = kBig16 && kPParts == 2 ? 1 : 2;         // f16 K buffers
  static constexpr uint32_t kHalf16 = kT * D * 2;                      // one f16 tile (K or V)
  static constexpr uint32_t kOff8 = 0;                        // the staging rings: K, then V
  static constexpr uint32_t kOffK8 = 0, kOffV8 = kStK * kStage, kOff16 = kOffV8 + kStV * kStage;
  static constexpr uint32_t kOffP = kOff16 + (kNK16 + 1) * kHalf16;   // f16 stage: K buffer(s) | V
  static constexpr uint32_t kPPart = 128 * 128;               // P: 128 rows x 64 tokens, 16-bit
  static constexpr uint32_t kPBuf = kPPart * kPParts;         // (bf16 V: high part | low part)
  static constexpr uint32_t kOffMeta = kOffP + 2 * kPBuf;     // meta ring: 4 tiles
  static constexpr uint32_t kOffX = kOffMeta + 4 * kMeta;     // exchange floats (see xf below)
  static constexpr uint32_t kOffBar = kOffX + 8 * 128 * 4 + 64;
  static constexpr uint32_t kOffMisc = kOffBar + 32 * 8;
  static constexpr uint32_t kOffList = kOffMisc + 64;         // work list + its scan scratch
  static constexpr uint32_t kSmem = kOffList + kListWords * 4 + 1024;   // + alignment slack
  static_assert(kSmem <= 232448, "shared memory");
  static_assert(kStage % 1024 == 0 && kOff16 % 1024 == 0 && kOffP % 1024 == 0 && kOffMeta % 16 == 0 &&
                    kOffBar % 8 == 0, "alignment");
  static_assert(8 * 32 * kEpiStride * 4 <= kOffP, "output staging fits in the staging ring and f16 stage");
};

// mbarriers (8 bytes each), named by their shared-memory address. K and V are staged in rings
// of their own, so a K stage is free again as soon as its K is widened while the V stage waits
// for its V. The f16 stage has two K buffers and one V buffer: K(j) may be widened once the
// QK^T of tile j - 2 is done, V(j) once the PV of tile j - 1 is done.
struct BarsI8 {
  uint32_t base;
  __device__ uint32_t at(uint32_t i) const { return base + 8u * i; }
  __device__ uint32_t fullK8(int s) const { return at(0 + s); }    // staged K tile landed
  __device__ uint32_t emptyK8(int s) const { return at(2 + s); }   // converters done with it
  __device__ uint32_t fullV8(int s) const { return at(4 + s); }    // staged V tile landed
  __device__ uint32_t emptyV8(int s) const { return at(7 + s); }   // converters done with it
  __device__ uint32_t fullK16(int b) const { return at(10 + b); }  // f16 K buffer b written
  __device__ uint32_t emptyK16(int b) const { return at(12 + b); } // its QK^T is done
  __device__ uint32_t fullV16() const { return at(14); }           // f16 V written
  __device__ uint32_t emptyV16() const { return at(15); }          // its PV is done
  __device__ uint32_t s_full(int s) const { return at(16 + s); }   // QK^T into S buffer s done
  __device__ uint32_t s_free(int s) const { return at(18 + s); }   // S buffer s read
  __device__ uint32_t p_full(int s) const { return at(20 + s); }   // P buffer s written (O rescaled)
  __device__ uint32_t pv_done(int s) const { return at(22 + s); }  // PV from P buffer s done
  __device__ uint32_t q_full() const { return at(24); }            // Q in TMEM
  __device__ uint32_t mma_fin() const { return at(25); }           // final commits of both issuers
  __device__ uint32_t meta_full(int s) const { return at(26 + s); }  // meta ring slot s written
};

__device__ __forceinline__ void set_abort_i8(uint32_t abort, uint32_t* status) {
  if (!ld_volatile_shared(abort)) {
    asm volatile("st.volatile.shared.b32 [%0], %1;" ::"r"(abort), "r"(1) : "memory");
    atomicOr(status, TLLM_FLAG_TIMEOUT);
  }
}

// byte offset of (row, byte) inside a [rows][128 B] block in the 128-byte swizzle layout
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t byte) {
  return (row >> 3) * 1024 + (row & 7) * 128 + ((((byte >> 4) ^ row) & 7) << 4) + (byte & 15);
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// V layouts, each a separate instance: token-major, dimension-major ([pages, Hkv, D, bs]), and
// dimension-major with 8-byte dim rows (8-token pages of an 8-bit cache)
constexpr int kVTok = 0, kVDim = 1, kVDim8 = 2;

// kKv: the cache's element type (kKvI8, kKvE4m3, kKvF16 or kKvBf16); kVL: the V layout
template <int D, int kKv, int kVL>
__global__ void __launch_bounds__(kThreads)
    partial_tc_i8_kernel(const Params p, const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap) {
  constexpr bool k16 = kKv == kKvF16 || kKv == kKvBf16;   // 16-bit cache: no per-token scales
  constexpr bool kVdm = kVL != kVTok;
  constexpr int kEsz = k16 ? 2 : 1;
  constexpr int kPParts = kKv == kKvBf16 ? 2 : 1;          // bf16 V: P as high + low bf16 parts
  using S = Lay<D, kEsz, kPParts>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) pdl_launch_dependents();
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S::kOffMisc);
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  int* wlist = reinterpret_cast<int*>(sm + S::kOffList);
  const BarsI8 bars{sbase + S::kOffBar};
  const uint32_t abort = sbase + S::kOffMisc + 4;
  const int bs = p.bs, bs_sh = __ffs(bs) - 1;
  const int brows = bs < kT ? bs : kT;                     // rows of one TMA box
  const int ppt = bs < kT ? kT >> bs_sh : 1;               // pages a tile touches
  // exchange floats of the two threads of a row: [0, 512) tile row maxima [parity][half][row],
  // [512, 768) query maxima [half][row], [768, 1024) row sums [half][row]; [1024, 1028) the
  // converter warps' tile maxima (bf16 K)
  float* xf = reinterpret_cast<float*>(sm + S::kOffX);

  // the real (request x kv head, split) items of the work list, in turn
  for (int round0 = 0;; round0 += kListCap) {
  const int n_list = build_work_list(p, wlist, round0);
  for (int li = 0; li < n_list; li++) {
  const int u = wlist[li] >> 8, b = u / p.Hkv, g = u % p.Hkv, split = wlist[li] & 255;
  const int raw_ctx = p.context_lens[b];
  const int ctx = clamp_ctx(raw_ctx, p.max_ctx);
  if (raw_ctx != ctx && tid == 0 && split == 0) atomicOr(p.status, TLLM_FLAG_CTX_CLAMPED);
  const Span sp = request_span(ctx, p.Lq, p.window, p.num_splits, p.min_chunk, p.align);
  if (split >= sp.nsplit) continue;
  const int t0 = sp.base + split * sp.chunk;
  const int t1 = min(ctx, t0 + sp.chunk);
  const int vlo = max(t0, sp.lo);
  const int n_tiles = t1 > t0 ? (t1 - t0 + kT - 1) / kT : 0;
  const bool finalize = sp.nsplit == 1;
  const int u_split = u * p.max_splits + split;

  if (n_tiles == 0) {                                      // nothing visible: zero rows
    for (int idx = tid; idx < p.R * D; idx += kThreads) {
      const int r = idx / D, d = idx % D;
      if (finalize) {
        const int i = r / p.G, hq = g * p.G + r % p.G;
        store_f32(p.out, p.out_dtype, ((int64_t)(b * p.Lq + i) * p.Hq + hq) * D + d, 0.f);
      } else {
        store_rec(p, ((int64_t)u_split * p.R + r) * D + d, 0.f);
        if (d == 0) p.ws_lse[(int64_t)u_split * p.R + r] = -INFINITY;
      }
    }
    continue;
  }

  if (tid == 0) {
    for (int s = 0; s < S::kStK; s++) {
      mbar_init(bars.fullK8(s), 1 + 32 + 1);               // expect_tx + 32 lanes' scale copies + mask
      mbar_init(bars.emptyK8(s), 4);                       // one elected lane per converter warp
    }
    for (int s = 0; s < S::kStV; s++) {
      mbar_init(bars.fullV8(s), 1 + 32 + 1);
      mbar_init(bars.emptyV8(s), 4);
    }
    for (int k = 0; k < 2; k++) {
      mbar_init(bars.fullK16(k), 4);                       // one elected lane per converter warp
      mbar_init(bars.emptyK16(k), 1);
    }
    mbar_init(bars.fullV16(), 4);
    mbar_init(bars.emptyV16(), 1);
    for (int s = 0; s < 2; s++) {
      mbar_init(bars.s_full(s), 1);
      mbar_init(bars.s_free(s), 8);                        // one elected lane per softmax warp
      mbar_init(bars.p_full(s), 8);
      mbar_init(bars.pv_done(s), 1);
    }
    for (int s = 0; s < 4; s++) mbar_init(bars.meta_full(s), 4);
    mbar_init(bars.q_full(), 8);
    mbar_init(bars.mma_fin(), 2);
    *reinterpret_cast<volatile int*>(sm + S::kOffMisc + 4) = 0;
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 0 || warp == 2) {
    // ---------------- producers: warp 0 the K tiles, warp 2 the V tiles ----------------
    const bool isk = warp == 0;
    const int nst = isk ? S::kStK : S::kStV;
    const uint32_t ring = isk ? S::kOffK8 : S::kOffV8;
    auto full = [&](int st) { return isk ? bars.fullK8(st) : bars.fullV8(st); };
    auto empty = [&](int st) { return isk ? bars.emptyK8(st) : bars.emptyV8(st); };
    // page id of slot `lane` of tile jt (-1: not read / invalid); read one tile ahead
    auto page_of = [&](int jt) -> int {
      if (jt >= n_tiles || lane >= ppt) return -1;
      const int tt = t0 + jt * kT, first = bs < kT ? tt + lane * bs : tt;
      const int last = bs < kT ? first + bs : tt + kT;
      if (max(first, sp.lo) >= min(last, t1)) return -1;
      const int pg = page_at(p, b, first >> bs_sh);
      if (pg < 0 || pg >= p.num_pages) {
        if (isk) atomicOr(p.status, TLLM_FLAG_BAD_PAGE);
        return -1;
      }
      return pg;
    };
    int pg_next = page_of(0);
    int issued = 0;
    for (int j = 0; j < n_tiles; j++) {
      const int st = j % nst;
      if (j >= nst && !mbar_wait(empty(st), ((j / nst) - 1) & 1, abort)) set_abort_i8(abort, p.status);
      if (ld_volatile_shared(abort)) break;
      const int pg = pg_next;
      pg_next = page_of(j + 1);
      const int tt = t0 + j * kT;
      const uint32_t mask = __ballot_sync(kFull, pg >= 0);
      const uint32_t stg = sbase + ring + st * S::kStage;
      if (lane == 0) mbar_arrive_expect_tx(full(st), __popc(mask) * (uint32_t)brows * D * kEsz);
      __syncwarp();
      if (pg >= 0) {
        if (isk || !kVdm) {
          const int row = (int)(((int64_t)pg * p.Hkv + g) * bs + (bs > kT ? (tt & (bs - 1)) : 0));
          tma_load_2d(stg + lane * brows * D * kEsz, isk ? &kmap : &vmap, 0, row, full(st));
        } else if (kVL == kVDim) {
          // a dimension-major V page: one box of D rows (dims) x brows tokens, staged as
          // [D][brows] behind the page slots before it
          tma_load_2d(stg + lane * brows * D * kEsz, &vmap, bs > kT ? (tt & (bs - 1)) : 0,
                      (int)(((int64_t)pg * p.Hkv + g) * D), full(st));
        } else {
          // 8-token pages of an 8-bit cache (8-byte dim rows, narrower than a box may be): the
          // page's D x 8 contiguous bytes in one plain bulk copy
          bulk_load(stg + lane * brows * D * kEsz,
                    static_cast<const uint8_t*>(p.v_cache) + ((int64_t)pg * p.Hkv + g) * D * bs * kEsz,
                    (uint32_t)(brows * D * kEsz), full(st));
        }
      }
      // scales (quantised caches): lanes 0..15 copy the scales of tokens 4l..4l+3; every lane
      // arrives once its copy (if any) has landed
      {
        if constexpr (!k16) {
          const int tk = 4 * (lane & 15);
          const int slot = bs < kT ? tk >> bs_sh : 0;
          const int pgl = __shfl_sync(kFull, pg, slot);
          const bool ok = pgl >= 0 && lane < 16;
          const int64_t srow = ok ? ((int64_t)pgl * p.Hkv + g) * bs + ((tt + tk) & (bs - 1)) : 0;
          if (lane < 16) cp_async16(stg + S::kRaw + tk * 4, (isk ? p.k_scales : p.v_scales) + srow, ok ? 16u : 0u);
        }
        cp_async_arrive_noinc(full(st));
      }
      if (lane == 0) {
        *reinterpret_cast<volatile uint32_t*>(sm + ring + st * S::kStage + S::kRaw + S::kScT) = mask;
        mbar_arrive(full(st));
      }
      issued = j + 1;
    }
    // drain: every issued stage's copies land before the item ends
    for (int j = max(0, issued - nst); j < issued; j++)
      if (!mbar_wait(full(j % nst), (j / nst) & 1, 0u)) set_abort_i8(abort, p.status);
  } else if (warp == 1 || warp == 3) {
    // ---------------- MMA issuers: warp 1 every QK^T, warp 3 every PV (one thread each) ----------------
    if (lane == 0) {
      bool ok = true;
      if (warp == 1) {
        const uint32_t idqk = idesc_f16(128, kT, 0, 0, 0);   // Q and K in f16
        ok = mbar_wait(bars.q_full(), 0, abort);
        // (a failure-detection test stalls here: no QK^T, so every wait on S runs out)
        for (int j = 0; ok && j < n_tiles && !p.test_stall; j++) {
          const int sb = j & 1;                            // S buffer (and f16 K buffer) of tile j
          const int kb = S::kNK16 == 2 ? sb : 0;
          if (!mbar_wait(bars.fullK16(kb), (S::kNK16 == 2 ? j >> 1 : j) & 1, abort)) { ok = false; break; }
          if (j >= 2 && !mbar_wait(bars.s_free(sb), ((j >> 1) - 1) & 1, abort)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kt = sbase + S::kOff16 + kb * S::kHalf16;
#pragma unroll
          for (int k = 0; k < D / 16; k++)
            mma_f16_ts(tmem + kColS + 64 * sb, tmem + kColQ + 8 * k,
                       sdesc_sw128(kt + (k >> 2) * S::kAtom + 32 * (k & 3), 16, 1024), idqk, k > 0 ? 1u : 0u);
          mma_commit(bars.s_full(sb));
          mma_commit(bars.emptyK16(kb));
        }
      } else {
        // P and V in f16 (bf16 V: both bf16); V MN-major as widened from token-major pages, K-major
        // (8-token blocks of D rows x 16 bytes) from dimension-major ones
        const uint32_t idpv = idesc_f16(128, D, kPParts - 1, 0, kVdm ? 0 : 1);
        const uint32_t vt = sbase + S::kOff16 + S::kNK16 * S::kHalf16;
        for (int j = 0; ok && j < n_tiles; j++) {
          const int pb = j & 1;
          if (!mbar_wait(bars.p_full(pb), (j >> 1) & 1, abort)) { ok = false; break; }
          if (!mbar_wait(bars.fullV16(), j & 1, abort)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kT / 16; k++)
#pragma unroll
            for (int part = 0; part < kPParts; part++)
              mma_f16_ss(tmem + kColO,
                         sdesc_sw128(sbase + S::kOffP + pb * S::kPBuf + part * S::kPPart + 32 * k, 16, 1024),
                         kVdm ? sdesc_none(vt + 32 * D * k, 16 * D, 128) : sdesc_sw128(vt + 2048 * k, S::kAtom, 1024),
                         idpv, (j > 0 || k > 0 || part > 0) ? 1u : 0u);
          mma_commit(bars.pv_done(pb));
          mma_commit(bars.emptyV16());
        }
      }
      if (!ok) set_abort_i8(abort, p.status);
      // every MMA issued must finish before the item ends (both issuers commit here)
      mma_commit(bars.mma_fin());
      if (!mbar_wait(bars.mma_fin(), 0, 0u)) set_abort_i8(abort, p.status);
    }
    // lanes 1..31 wait here for lane 0, so that the warp reaches the item's closing CTA barrier
    // (an aligned barrier) converged
    __syncwarp();
  } else if (warp >= 12) {
    // ---------------- converters: staged tiles -> f16 tiles, scales and mask ----------------
    // Warps 12..15 widen, all four on each, K(0), then for every later step j K(j) and V(j - 1),
    // then the last V: K(j) into f16 K buffer j % 2 once the QK^T of tile j - 2 is done, V(j)
    // into the f16 V buffer once the PV of tile j - 1 is done. K thus runs a tile ahead of V,
    // and the QK^T of tile j + 1 goes out while the softmax of tile j runs.
    const int ct = tid - 384;                              // 0..127
    constexpr int kEpc = 16 / kEsz;                        // elements per 16-byte chunk
    constexpr int kChunksPerRow = D / kEpc, kPer = kT * kChunksPerRow / 128;
    float* xc = xf + 1024;                                 // the converter warps' tile maxima (bf16 K)
    for (int step = 0; step <= n_tiles; step++) {
#pragma unroll
      for (int which = 0; which < 2; which++) {            // 0: K of tile step, 1: V of tile step - 1
        const int j = step - which;
        if (which == 0 ? j >= n_tiles : j < 0) continue;
        const int stk = j % S::kStK, stv = j % S::kStV;
        const uint8_t* srck = sm + S::kOffK8 + stk * S::kStage;
        const uint8_t* srcv = sm + S::kOffV8 + stv * S::kStage;
        if (which == 0) {
          if (!mbar_wait(bars.fullK8(stk), (j / S::kStK) & 1, abort)) set_abort_i8(abort, p.status);
          if constexpr (!S::kBig16)
            if (!mbar_wait(bars.fullV8(stv), (j / S::kStV) & 1, abort)) set_abort_i8(abort, p.status);
        }
        if constexpr (S::kBig16)                           // (one-deep V ring: V(j) lands after V(j - 1) is widened)
          if (which == 1 && !mbar_wait(bars.fullV8(stv), (j / S::kStV) & 1, abort)) set_abort_i8(abort, p.status);
        const uint8_t* src = which == 0 ? srck : srcv;     // (the K stage is not read for V: it may hold tile j + 2)
        const uint32_t pmask8 = *reinterpret_cast<const volatile uint32_t*>(src + S::kRaw + S::kScT);
        const int tt = t0 + j * kT;
        // is row t of this tile a token the split reads? (a slot past the context, before the
        // window, or of a page not loaded holds stale or poisoned bytes)
        auto read_tok = [&](int t) -> bool {
          const int slot = bs < kT ? t >> bs_sh : 0;
          return ((pmask8 >> slot) & 1) && tt + t >= vlo && tt + t < t1;
        };
        // this thread's chunks of the operand, loaded before anything is converted (their
        // latencies overlap); a 16-bit tile of head_dim 256 (16 chunks a thread) is loaded and
        // stored below in two batches of 8, within the register budget
        constexpr int kBatch = S::kBig16 ? 8 : kPer;
        uint4 w[kBatch];
        if constexpr (!S::kBig16)
#pragma unroll
        for (int i = 0; i < kPer; i++) {
          const int c = ct + 128 * i, t = c / kChunksPerRow, d0 = (c % kChunksPerRow) * kEpc;
          // (a dimension-major V stage holds the same bytes in the order page slot, dim, token:
          // chunk c is the c-th 16 bytes of it)
          w[i] = *reinterpret_cast<const uint4*>(src + (kVdm && which == 1 ? 16 * c : (t * D + d0) * kEsz));
        }
        // A bf16 K tile enters f16 scaled by 2^e, e from the largest |x| the split reads in it,
        // so that this maximum lies in [2^13, 2^14): every element within 2^-27 of it converts to
        // a normal f16 exactly (bf16 keeps 8 significant bits, f16 11); a smaller one rounds by
        // at most 2^-38 of the maximum, below the fp32 rounding bound of the score it enters.
        // 2^-e goes to the tile's per-token K scales. An f16 tile, and a bf16 V tile, is copied
        // as it is (e = 0).
        int e = 0;
        if (kKv == kKvBf16 && which == 0) {
          float mx = 0.f;
#pragma unroll
          for (int i = 0; i < kPer; i++) {
            const int t = (ct + 128 * i) / kChunksPerRow;
            if (read_tok(t)) {
              uint4 x;
              if constexpr (S::kBig16)
                x = *reinterpret_cast<const uint4*>(src + (t * D + ((ct + 128 * i) % kChunksPerRow) * kEpc) * kEsz);
              else
                x = w[i];
              const uint32_t ws[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int k = 0; k < 4; k++)
                mx = fmax3(mx, fabsf(__uint_as_float(ws[k] << 16)), fabsf(__uint_as_float(ws[k] & 0xffff0000u)));
            }
          }
          mx = warp_max_abs(isfinite(mx) ? mx : 0.f);
          if (lane == 0) xc[warp - 12] = mx;
          named_bar(2, 128);                               // the four converter warps
          mx = fmaxf(fmaxf(xc[0], xc[1]), fmaxf(xc[2], xc[3]));
          named_bar(2, 128);                               // all read before the next tile's write
          if (mx > 0.f) e = min(125, max(-125, 14 - exponent_of(mx)));
        }
        if (which == 0) {
          // The tile's meta, into ring slot j % 4: scales (thread ct: the K scale of token ct
          // for ct < 64, else the V scale of token ct - 64), the page mask and the tile's
          // largest |V scale|. The K scales leave here multiplied by the softmax scale in log2
          // units, so that a score reaches the softmax as one product with the query row's
          // power of two, which is exact. Slot j % 4 last held tile j - 4, whose softmax is
          // over: V(j - 3), widened two steps before this one, waited for the PV of tile j - 4,
          // which waited for that softmax. A token the split does not read gets zero scales (its
          // staged scale may be stale or NaN), so that the softmax's P x V-scale product is 0
          // there without a select.
          float scv;
          if constexpr (k16) scv = ct < kT ? __int_as_float((127 - e) << 23) : 1.f;   // 2^-e for K
          else scv = reinterpret_cast<const float*>((ct < kT ? srck : srcv) + S::kRaw)[ct & (kT - 1)];
          if (!read_tok(ct & (kT - 1))) scv = 0.f;
          uint8_t* meta = sm + S::kOffMeta + (j & 3) * S::kMeta;
          reinterpret_cast<float*>(meta)[ct] = ct < kT ? scv * p.scale_log2 : scv;
          const float vm = warp_max_abs(ct >= kT && isfinite(scv) ? scv : 0.f);
          if (ct == 0) *reinterpret_cast<uint32_t*>(meta + S::kSc) = pmask8;
          if (lane == 0 && ct >= kT) reinterpret_cast<float*>(meta + S::kSc + 4)[(ct - kT) >> 5] = vm;
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.meta_full(j & 3));
        }
        // f16 K buffer j % 2 is free once the QK^T of tile j - 2 is done (with one K buffer: of
        // tile j - 1); the V buffer once the PV of tile j - 1 is done
        const int kb = S::kNK16 == 2 ? (j & 1) : 0;        // (K) its f16 buffer
        if (which == 0 ? (j >= S::kNK16 && !mbar_wait(bars.emptyK16(kb), (S::kNK16 == 2 ? (j >> 1) - 1 : j - 1) & 1,
                                                      abort))
                       : (j >= 1 && !mbar_wait(bars.emptyV16(), (j - 1) & 1, abort)))
          set_abort_i8(abort, p.status);
        const uint32_t dst = sbase + S::kOff16 + (which == 0 ? kb : S::kNK16) * S::kHalf16;
        const __half2 bias = __half2(__half_raw{0x6480}, __half_raw{0x6480});
        const float emul = __int_as_float((e + 127) << 23);
        if constexpr (S::kBig16) {
          // a 16-bit tile of head_dim 256 (token-major V only): the same copy as below, in two
          // batches of 8 chunks a thread
#pragma unroll
          for (int b0 = 0; b0 < kPer; b0 += kBatch) {
#pragma unroll
            for (int i = 0; i < kBatch; i++) {
              const int c = ct + 128 * (b0 + i), t = c / kChunksPerRow, d0 = (c % kChunksPerRow) * kEpc;
              w[i] = *reinterpret_cast<const uint4*>(src + (t * D + d0) * kEsz);
            }
#pragma unroll
            for (int i = 0; i < kBatch; i++) {
              const int c = ct + 128 * (b0 + i), t = c / kChunksPerRow, d0 = (c % kChunksPerRow) * kEpc;
              const bool ok = which == 0 || read_tok(t);   // (V rows of unread tokens become zero)
              const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
              const uint32_t base = dst + (d0 >> 6) * S::kAtom;
              const uint32_t byte = (d0 & 63) * 2;
              uint32_t h[4];
#pragma unroll
              for (int q = 0; q < 4; q++) {
                if (kKv == kKvBf16 && which == 0) {
                  const __half2 v2 = __floats2half2_rn(__uint_as_float(ws[q] << 16) * emul,
                                                       __uint_as_float(ws[q] & 0xffff0000u) * emul);
                  h[q] = *reinterpret_cast<const uint32_t*>(&v2);
                } else {
                  h[q] = ok ? ws[q] : 0u;
                }
              }
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(base + swz(t, byte)), "r"(h[0]),
                           "r"(h[1]), "r"(h[2]), "r"(h[3]));
            }
          }
        } else if (kVdm && which == 1) {
          // dimension-major V: chunk c holds kEpc tokens of one dim of one page slot; widened,
          // they go to the K-major f16 V buffer, whose 8-token blocks are D rows x 16 bytes.
          // Tokens the split does not read are zeroed element by element (e4m3 and 16-bit codes
          // may be NaN there; int8 is always finite).
          if constexpr (kVL == kVDim8) {
            // 8-token pages of an 8-bit cache: chunk c holds the 8-token rows of dims d and
            // d + 1 of page slot c / (D / 2); their widened rows are adjacent in the V buffer
            constexpr int kDsh = D == 64 ? 6 : D == 128 ? 7 : 8;
#pragma unroll
            for (int i = 0; i < kPer; i++) {
              const int c = ct + 128 * i, d = (c & (D / 2 - 1)) * 2, t0c = (c >> (kDsh - 1)) << 3;
              const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
              uint32_t h[8];
              if constexpr (kKv == kKvE4m3) {
#pragma unroll
                for (int q = 0; q < 8; q++) {
                  h[q] = e4m3x2_to_f16x2((uint16_t)(ws[q >> 1] >> (16 * (q & 1))));
                  const int tq = t0c + 2 * (q & 3);
                  h[q] &= (read_tok(tq) ? 0x0000ffffu : 0u) | (read_tok(tq + 1) ? 0xffff0000u : 0u);
                }
              } else {
#pragma unroll
                for (int q = 0; q < 8; q++) {
                  const uint32_t x = __byte_perm(ws[q >> 1] ^ 0x80808080u, 0x64646464u, (q & 1) ? 0x5342u : 0x5140u);
                  const __half2 v2 = __hsub2(*reinterpret_cast<const __half2*>(&x), bias);
                  h[q] = *reinterpret_cast<const uint32_t*>(&v2);
                }
              }
              const uint32_t a0 = dst + (t0c >> 3) * (16 * D) + 16 * d;
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a0), "r"(h[0]), "r"(h[1]), "r"(h[2]),
                           "r"(h[3]));
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a0 + 16), "r"(h[4]), "r"(h[5]), "r"(h[6]),
                           "r"(h[7]));
            }
          } else {
            // (all powers of two: a page slot's dim row is 2^csh chunks, a slot D << csh chunks)
            constexpr int kDsh = D == 64 ? 6 : D == 128 ? 7 : 8, kEsh = kEsz == 2 ? 3 : 4;
            const int bsh = bs_sh < 6 ? bs_sh : 6, csh = bsh - kEsh;
#pragma unroll
            for (int i = 0; i < kPer; i++) {
              const int c = ct + 128 * i, rem = c & ((D << csh) - 1), d = rem >> csh;
              const int t0c = ((c >> (kDsh + csh)) << bsh) + ((rem & ((1 << csh) - 1)) << kEsh);   // first token
              const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
              uint32_t h[8];
              if constexpr (!k16) {
                if constexpr (kKv == kKvE4m3) {
#pragma unroll
                  for (int q = 0; q < 8; q++) h[q] = e4m3x2_to_f16x2((uint16_t)(ws[q >> 1] >> (16 * (q & 1))));
                } else {
#pragma unroll
                  for (int q = 0; q < 8; q++) {
                    const uint32_t x = __byte_perm(ws[q >> 1] ^ 0x80808080u, 0x64646464u, (q & 1) ? 0x5342u : 0x5140u);
                    const __half2 v2 = __hsub2(*reinterpret_cast<const __half2*>(&x), bias);
                    h[q] = *reinterpret_cast<const uint32_t*>(&v2);
                  }
                }
              } else {
#pragma unroll
                for (int q = 0; q < 4; q++) h[q] = ws[q];
              }
              if constexpr (kKv != kKvI8) {
#pragma unroll
                for (int q = 0; q < kEpc / 2; q++)
                  h[q] &= (read_tok(t0c + 2 * q) ? 0x0000ffffu : 0u) | (read_tok(t0c + 2 * q + 1) ? 0xffff0000u : 0u);
              }
              const uint32_t a0 = dst + (t0c >> 3) * (16 * D) + 16 * d;
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a0), "r"(h[0]), "r"(h[1]), "r"(h[2]),
                           "r"(h[3]));
              if constexpr (!k16)
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a0 + 16 * D), "r"(h[4]), "r"(h[5]),
                             "r"(h[6]), "r"(h[7]));
            }
          }
        } else {
#pragma unroll
        for (int i = 0; i < kPer; i++) {
          const int c = ct + 128 * i, t = c / kChunksPerRow, d0 = (c % kChunksPerRow) * kEpc;
          // V rows of tokens the split does not read become zero: their bytes may be NaN (an
          // e4m3 or 16-bit code), and the PV MMA would carry 0 x NaN. (K needs no such care:
          // the softmax selects -inf for those tokens' scores.) Int8 codes are always finite.
          const bool ok = kKv == kKvI8 || which == 0 || read_tok(t);
          const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
          const uint32_t base = dst + (d0 >> 6) * S::kAtom;
          const uint32_t byte = (d0 & 63) * 2;
          if constexpr (!k16) {
            uint32_t h[8];
            if constexpr (kKv == kKvE4m3) {
              // two e4m3 codes -> f16x2, element 0 (the lower byte) in the low half
#pragma unroll
              for (int q = 0; q < 8; q++) h[q] = ok ? e4m3x2_to_f16x2((uint16_t)(ws[q >> 1] >> (16 * (q & 1)))) : 0u;
            } else {
              // int8 -> f16 exactly: the byte, sign bit flipped, placed under the f16 exponent
              // of 1024 reads 1024 + (x + 128); subtracting 1152 leaves x
#pragma unroll
              for (int q = 0; q < 8; q++) {
                const uint32_t x = __byte_perm(ws[q >> 1] ^ 0x80808080u, 0x64646464u, (q & 1) ? 0x5342u : 0x5140u);
                const __half2 v2 = __hsub2(*reinterpret_cast<const __half2*>(&x), bias);
                h[q] = *reinterpret_cast<const uint32_t*>(&v2);
              }
            }
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(base + swz(t, byte)), "r"(h[0]), "r"(h[1]),
                         "r"(h[2]), "r"(h[3]));
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(base + swz(t, byte + 16)), "r"(h[4]),
                         "r"(h[5]), "r"(h[6]), "r"(h[7]));
          } else {
            uint32_t h[4];
#pragma unroll
            for (int q = 0; q < 4; q++) {
              if (kKv == kKvBf16 && which == 0) {
                const __half2 v2 = __floats2half2_rn(__uint_as_float(ws[q] << 16) * emul,
                                                     __uint_as_float(ws[q] & 0xffff0000u) * emul);
                h[q] = *reinterpret_cast<const uint32_t*>(&v2);
              } else {
                h[q] = ok ? ws[q] : 0u;
              }
            }
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(base + swz(t, byte)), "r"(h[0]), "r"(h[1]),
                         "r"(h[2]), "r"(h[3]));
          }
        }
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(which == 0 ? bars.fullK16(kb) : bars.fullV16());
          mbar_arrive(which == 0 ? bars.emptyK8(stk) : bars.emptyV8(stv));
        }
      }
    }
    // the releases of the f16 buffers by the last tiles' MMAs (asynchronous tcgen05.commit
    // arrivals) must have landed before the next item re-initialises the barriers
    const int nl = n_tiles - 1;
    if constexpr (S::kNK16 == 2) {
      if (!mbar_wait(bars.emptyK16(nl & 1), (nl >> 1) & 1, abort)) set_abort_i8(abort, p.status);
      if (nl >= 1 && !mbar_wait(bars.emptyK16((nl - 1) & 1), ((nl - 1) >> 1) & 1, abort))
        set_abort_i8(abort, p.status);
    } else {
      if (!mbar_wait(bars.emptyK16(0), nl & 1, abort)) set_abort_i8(abort, p.status);
    }
    if (!mbar_wait(bars.emptyV16(), nl & 1, abort)) set_abort_i8(abort, p.status);
  } else if (warp >= 4) {
    // ---------------- softmax: two threads per packed row r (TMEM lane), one per token half ----------------
    const int hh = (warp - 4) >> 2;                        // token half (0: tokens 0..31, 1: 32..63)
    const int r = 32 * (warp & 3) + lane;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const bool real = r < p.R;
    const int qi = real ? r / p.G : 0, qh = g * p.G + (real ? r % p.G : 0);
    const int pos = real ? ctx - p.Lq + qi : -1;
    // Q row -> TMEM columns [0, D/2) in f16, two elements per column (even element low); this
    // thread converts elements [hh D/2, (hh + 1) D/2). A bf16 row is first scaled by 2^e so that
    // its largest |q| lies in [2^13, 2^14): every element that is at least 2^-14 after scaling
    // converts exactly (bf16 carries 8 significant bits, f16 11); a smaller one rounds by at most
    // 2^-25, far below the fp32 rounding of a score whose largest term is near 2^13 |k|. The
    // scores are scaled back by qscale = 2^-e, a power of two, so the row maximum in log2 units
    // is exact and the largest term of every row's exponent sum is exactly 2^C, however large
    // the scores.
    float qscale = 1.f;
    {
      const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                         ((int64_t)(b * p.Lq + qi) * p.Hq + qh) * D + hh * (D / 2));
      const bool qbf = p.q_dtype == TLLM_BF16;
      // the thread's half row is loaded at once (one memory round trip; it is on the path to
      // the first QK^T)
      uint4 qv[D / 16];
#pragma unroll
      for (int c = 0; c < D / 16; c++) qv[c] = real ? __ldg(qsrc + c) : make_uint4(0, 0, 0, 0);
      float emul = 1.f;
      if (qbf) {
        float mx = 0.f;
#pragma unroll
        for (int c = 0; c < D / 16; c++) {
          const uint32_t xs[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
#pragma unroll
          for (int k = 0; k < 4; k++)
            mx = fmax3(mx, fabsf(__uint_as_float(xs[k] << 16)), fabsf(__uint_as_float(xs[k] & 0xffff0000u)));
        }
        // the row's largest |q| over both halves
        xf[512 + 128 * hh + r] = mx;
        named_bar(1, kSmThreads);
        mx = fmaxf(xf[512 + r], xf[640 + r]);
        int e = 0;
        if (mx > 0.f && mx <= 3.402823466e38f) {
          int ex;
          frexpf(mx, &ex);
          e = min(125, max(-125, 14 - ex));
        }
        emul = __int_as_float((e + 127) << 23);
        qscale = __int_as_float((127 - e) << 23);
      }
#pragma unroll
      // this thread's D / 4 TMEM columns, 32 (or, for head_dim 64, 16) at a time
      constexpr int kQc = D / 4 < 32 ? D / 4 : 32;
#pragma unroll
      for (int c0 = 0; c0 < D / 4; c0 += kQc) {
        uint32_t w[kQc];
#pragma unroll
        for (int c = 0; c < kQc / 4; c++) {
          const uint4 x = qv[c0 / 4 + c];
          w[4 * c] = x.x;
          w[4 * c + 1] = x.y;
          w[4 * c + 2] = x.z;
          w[4 * c + 3] = x.w;
        }
        if (qbf) {
#pragma unroll
          for (int k = 0; k < kQc; k++) {
            const __half2 h2 = __floats2half2_rn(__uint_as_float(w[k] << 16) * emul,
                                                 __uint_as_float(w[k] & 0xffff0000u) * emul);
            w[k] = *reinterpret_cast<const uint32_t*>(&h2);
          }
        }
        if constexpr (kQc == 32) tmem_st32(tmem + lane_off + kColQ + hh * (D / 4) + c0, w);
        else tmem_st16(tmem + lane_off + kColQ + hh * (D / 4) + c0, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.q_full());
    }
    float M = -INFINITY, l = 0.f;                          // running max (log2 units), this half's sum (units of 2^-C)
    int C = 1 << 20;                                       // P scale exponent, unset
    float e0_run = 0.f;                                    // exponent offset of O and l
    int last = -1;
    for (int j = 0; j < n_tiles; j++) {
      last = j;
      const int sb = j & 1;
      const int tt = t0 + j * kT;
      const uint8_t* meta = sm + S::kOffMeta + (j & 3) * S::kMeta;
      const float* ksc = reinterpret_cast<const float*>(meta) + 32 * hh;
      const float* vsc = reinterpret_cast<const float*>(meta) + kT + 32 * hh;
      if (!mbar_wait(bars.meta_full(j & 3), (j >> 2) & 1, abort)) set_abort_i8(abort, p.status);
      const uint32_t pmask = *reinterpret_cast<const volatile uint32_t*>(meta + S::kSc);
      const float vmax = fmaxf(reinterpret_cast<const float*>(meta + S::kSc + 4)[0],
                               reinterpret_cast<const float*>(meta + S::kSc + 4)[1]);
      if (!mbar_wait(bars.s_full(sb), (j >> 1) & 1, abort)) set_abort_i8(abort, p.status);
      tc_fence_after();
      uint32_t sreg[32];
      tmem_ld32(tmem + lane_off + kColS + 64 * sb + 32 * hh, sreg);
      tmem_ld_wait(sreg);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.s_free(sb));

      // scores: u = raw x K scale (masked tokens -inf; their scales may be anything, NaN
      // included, so masking selects rather than multiplies). A tile every row sees whole (all
      // pages valid, every token read, at or before every row's position, inside its window)
      // takes no per-token mask.
      const float4* ks4 = reinterpret_cast<const float4*>(ksc);
      const float4* vs4 = reinterpret_cast<const float4*>(vsc);
      const uint32_t full_pages = ppt >= 32 ? kFull : ((1u << ppt) - 1u);
      const bool whole = pmask == full_pages && tt >= vlo && tt + kT <= t1 && tt + kT - 1 <= ctx - p.Lq &&
                         (p.window <= 0 || tt > ctx - 1 - p.window);
      float u[32];
      if (whole) {
#pragma unroll
        for (int i4 = 0; i4 < 8; i4++) {
          const float4 k4 = ks4[i4];
          const float2 a = fmul2(make_float2(__uint_as_float(sreg[4 * i4]), __uint_as_float(sreg[4 * i4 + 1])),
                                 make_float2(k4.x, k4.y));
          const float2 c = fmul2(make_float2(__uint_as_float(sreg[4 * i4 + 2]), __uint_as_float(sreg[4 * i4 + 3])),
                                 make_float2(k4.z, k4.w));
          u[4 * i4] = a.x;
          u[4 * i4 + 1] = a.y;
          u[4 * i4 + 2] = c.x;
          u[4 * i4 + 3] = c.y;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; i++) {
          const int ti = 32 * hh + i, t = tt + ti;
          const int slot = bs < kT ? ti >> bs_sh : 0;
          const bool vis = ((pmask >> slot) & 1) && t >= vlo && t < t1 && t <= pos &&
                           (p.window <= 0 || pos - t < p.window);
          u[i] = vis ? __uint_as_float(sreg[i]) * ksc[i] : -INFINITY;
        }
      }
      // rows past R see nothing (their scores stay -inf)
      if (!real) {
#pragma unroll
        for (int i = 0; i < 32; i++) u[i] = -INFINITY;
      }
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int k = 0; k < 16; k++) m4[k & 3] = fmax3(m4[k & 3], u[2 * k], u[2 * k + 1]);
      // the row maximum over both halves (slot by tile parity: the partner may still be reading
      // the previous tile's)
      float* xm = xf + 256 * sb;
      xm[128 * hh + r] = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
      named_bar(1, kSmThreads);
      const float mx = fmaxf(xm[r], xm[128 + r]);
      // P scale exponent C: vmax * 2^C < 2^(14 - kSlack); it only ever decreases (then O is
      // rescaled)
      if (vmax > 0.f) {
        int ex;
        frexpf(vmax, &ex);
        C = min(C, min(60, max(-60, 14 - kSlack - ex)));
      } else if (C == (1 << 20)) {
        C = 0;
      }
      // p' = 2^(u qscale + e0) with e0 = C - M (rounded): the row's largest term is at most
      // 2^(C + kSlack). O and l are kept in units of 2^-e0 for the e0 actually used, so its
      // rounding cancels in O / l and in the LSE (log2 l - e0), and a change of e0 rescales both
      // by 2^(e0 - e0_prev). Both threads of a row hold the same M, C and e0.
      const float M_new = mx * qscale > M + (float)kSlack ? mx * qscale : M;
      const float e0 = M_new == -INFINITY ? 0.f : (float)C - M_new;
      const float factor = M == -INFINITY ? (M_new == -INFINITY ? 1.f : 0.f) : ex2f(e0 - e0_run);
      e0_run = e0;
      const float2 qs2 = make_float2(qscale, qscale), e02 = make_float2(e0, e0);
      float2 ls = make_float2(0.f, 0.f);
      uint32_t pw[16];
      [[maybe_unused]] uint32_t pl[16];                    // bf16 V: the low parts of P
#pragma unroll
      for (int i4 = 0; i4 < 8; i4++) {
        const float4 v = vs4[i4];
        const float2 x01 = ffma2(make_float2(u[4 * i4], u[4 * i4 + 1]), qs2, e02);
        const float2 x23 = ffma2(make_float2(u[4 * i4 + 2], u[4 * i4 + 3]), qs2, e02);
        // u = -inf gives 2^-inf = 0; so does a row that has seen nothing yet (M_new = -inf,
        // e0 = 0, every u = -inf)
        const float2 p01 = make_float2(ex2f(x01.x), ex2f(x01.y)), p23 = make_float2(ex2f(x23.x), ex2f(x23.y));
        ls = fadd2(ls, fadd2(p01, p23));
        // (the V scale of a token the split does not read is 0, and its p is 0 too)
        const float2 w01 = fmul2(p01, make_float2(v.x, v.y)), w23 = fmul2(p23, make_float2(v.z, v.w));
        const float w0 = w01.x, w1 = w01.y, w2 = w23.x, w3 = w23.y;
        if constexpr (kPParts == 2) {
          const __nv_bfloat162 h01 = __floats2bfloat162_rn(w0, w1), h23 = __floats2bfloat162_rn(w2, w3);
          const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
          const __nv_bfloat162 l01 = __floats2bfloat162_rn(w0 - f01.x, w1 - f01.y);
          const __nv_bfloat162 l23 = __floats2bfloat162_rn(w2 - f23.x, w3 - f23.y);
          pw[2 * i4] = *reinterpret_cast<const uint32_t*>(&h01);
          pw[2 * i4 + 1] = *reinterpret_cast<const uint32_t*>(&h23);
          pl[2 * i4] = *reinterpret_cast<const uint32_t*>(&l01);
          pl[2 * i4 + 1] = *reinterpret_cast<const uint32_t*>(&l23);
        } else {
          const __half2 h01 = __floats2half2_rn(w0, w1), h23 = __floats2half2_rn(w2, w3);
          pw[2 * i4] = *reinterpret_cast<const uint32_t*>(&h01);
          pw[2 * i4 + 1] = *reinterpret_cast<const uint32_t*>(&h23);
        }
      }
      l = l * factor + (ls.x + ls.y);
      const float prev_M = M;
      M = M_new;

      // P buffer sb is free once the PV of tile j - 2 (which read it) is done
      if (j >= 2 && !mbar_wait(bars.pv_done(sb), ((j - 2) >> 1) & 1, abort)) set_abort_i8(abort, p.status);
      const uint32_t prow = sbase + S::kOffP + sb * S::kPBuf;
#pragma unroll
      for (int c = 0; c < 4; c++) {
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + swz(r, 64 * hh + 16 * c)),
                     "r"(pw[4 * c]), "r"(pw[4 * c + 1]), "r"(pw[4 * c + 2]), "r"(pw[4 * c + 3]));
        if constexpr (kPParts == 2)
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + S::kPPart + swz(r, 64 * hh + 16 * c)),
                       "r"(pl[4 * c]), "r"(pl[4 * c + 1]), "r"(pl[4 * c + 2]), "r"(pl[4 * c + 3]));
      }
      fence_proxy_async();
      // rescale this row of O (this thread: half of its columns) when its maximum grew or the P
      // scale shrank: O holds the tiles < j, so the PV of tile j - 1 must be done first
      const bool need = j >= 1 && factor != 1.f && prev_M != -INFINITY;
      if (__any_sync(kFull, need)) {
        if (!mbar_wait(bars.pv_done((j - 1) & 1), ((j - 1) >> 1) & 1, abort)) set_abort_i8(abort, p.status);
        tc_fence_after();
        const float f = need ? factor : 1.f;
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + kColO + hh * (D / 2) + c0, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; i++) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
          tmem_st32(tmem + lane_off + kColO + hh * (D / 2) + c0, o);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.p_full(sb));
    }

    // ---------------- epilogue: O / l (record or final output) ----------------
    // the last two PVs (one per P buffer): each commit's arrival lands before the item ends
    if (last >= 1 && !mbar_wait(bars.pv_done((last - 1) & 1), ((last - 1) >> 1) & 1, abort))
      set_abort_i8(abort, p.status);
    if (last >= 0 && !mbar_wait(bars.pv_done(last & 1), (last >> 1) & 1, abort)) set_abort_i8(abort, p.status);
    tc_fence_after();
    xf[768 + 128 * hh + r] = l;
    named_bar(1, kSmThreads);
    const float lt = xf[768 + r] + xf[896 + r];
    // (the TMEM loads are warp-collective: every lane takes part, only real rows store)
    const bool store = real && !ld_volatile_shared(abort);
    float mul = 0.f;
    // O and l are both in units of 2^-e0
    if (finalize) {
      if (lt > 0.f) mul = 1.f / (lt + (p.sinks ? ex2f(p.sinks[qh] * kLog2e + e0_run) : 0.f));
    } else {
      mul = lt > 0.f ? 1.f / lt : 0.f;
      if (store && hh == 0) p.ws_lse[(int64_t)u_split * p.R + r] = lt > 0.f ? log2f(lt) - e0_run : -INFINITY;
    }
    // O leaves through shared memory, 32 columns at a time: a thread holds one row, so storing
    // from registers would touch 32 rows per instruction; staged, each warp stores its own 32
    // rows as whole 128-byte lines. The staging ring and the f16 stage are free here: every
    // tile's copies landed and were widened before its PV, and its MMAs are done.
    float* stage = reinterpret_cast<float*>(sm + S::kOff8) + (warp - 4) * 32 * kEpiStride;
    const bool keep = !ld_volatile_shared(abort);
    // output row offset of this lane's row (-1: padding), computed once and shuffled to the
    // lanes that store it
    int64_t out_row = -1;
    if (r < p.R) out_row = ((int64_t)(b * p.Lq + r / p.G) * p.Hq + g * p.G + r % p.G) * D;
#pragma unroll 1
    for (int c0 = hh * (D / 2); c0 < (hh + 1) * (D / 2); c0 += 32) {
      uint32_t o[32];
      tmem_ld32(tmem + lane_off + kColO + c0, o);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(stage + lane * kEpiStride + i) =
            make_float4(__uint_as_float(o[i]) * mul, __uint_as_float(o[i + 1]) * mul,
                        __uint_as_float(o[i + 2]) * mul, __uint_as_float(o[i + 3]) * mul);
      __syncwarp();
      if (keep) {
        if (!finalize) {
          // lane: row 4k + lane / 8 of the warp's 32, columns c0 + 4 (lane % 8) .. + 3
#pragma unroll
          for (int k = 0; k < 8; k++) {
            const int rr = 4 * k + (lane >> 3), rg = 32 * (warp & 3) + rr;
            if (rg < p.R)
              store_rec4(p, ((int64_t)u_split * p.R + rg) * D + c0 + 4 * (lane & 7),
                         *reinterpret_cast<const float4*>(stage + rr * kEpiStride + 4 * (lane & 7)));
          }
        } else if (p.out_dtype == TLLM_F32) {
          // lane: row 4k + lane / 8 of the warp's 32, columns c0 + 4 (lane % 8) .. + 3
#pragma unroll
          for (int k = 0; k < 8; k++) {
            const int rr = 4 * k + (lane >> 3);
            const int64_t ob = __shfl_sync(kFull, out_row, rr);
            if (ob >= 0)
              *reinterpret_cast<float4*>(static_cast<float*>(p.out) + ob + c0 + 4 * (lane & 7)) =
                  *reinterpret_cast<const float4*>(stage + rr * kEpiStride + 4 * (lane & 7));
          }
        } else {
          // lane: row 8k + lane / 4 of the warp's 32, columns c0 + 8 (lane % 4) .. + 7 as one
          // 16-byte store
          const bool bf = p.out_dtype == TLLM_BF16;
#pragma unroll
          for (int k = 0; k < 4; k++) {
            const int rr = 8 * k + (lane >> 2);
            const int64_t ob = __shfl_sync(kFull, out_row, rr);
            const float4 x0 = *reinterpret_cast<const float4*>(stage + rr * kEpiStride + 8 * (lane & 3));
            const float4 x1 = *reinterpret_cast<const float4*>(stage + rr * kEpiStride + 8 * (lane & 3) + 4);
            uint32_t w[4];
            if (bf) {
              const __nv_bfloat162 h[4] = {__floats2bfloat162_rn(x0.x, x0.y), __floats2bfloat162_rn(x0.z, x0.w),
                                           __floats2bfloat162_rn(x1.x, x1.y), __floats2bfloat162_rn(x1.z, x1.w)};
              memcpy(w, h, 16);
            } else {
              const __half2 h[4] = {__floats2half2_rn(x0.x, x0.y), __floats2half2_rn(x0.z, x0.w),
                                    __floats2half2_rn(x1.x, x1.y), __floats2half2_rn(x1.z, x1.w)};
              memcpy(w, h, 16);
            }
            if (ob >= 0)
              *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + ob + c0 + 8 * (lane & 3)) =
                  make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();                                         // item done: every copy, MMA and TMEM access drained
  if (ld_volatile_shared(abort)) break;
  }
  if (n_list < kListCap || (n_list > 0 && ld_volatile_shared(abort))) break;
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder_i8() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D map over the cache viewed as [rows][inner elements of esz bytes], unswizzled (the
// converters read it row by row). Token-major: rows = pages * Hkv * bs, inner = D, a box one page
// (or one 64-token tile of a larger page). Dimension-major V: rows = pages * Hkv * D, inner = bs,
// a box D rows x box_inner tokens.
bool encode_i8_map(CUtensorMap* map, const void* base, int64_t rows, int inner, int box_rows, int esz,
                   int box_inner = 0) {
  auto enc = get_encoder_i8();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)inner * esz};
  cuuint32_t box[2] = {(cuuint32_t)(box_inner ? box_inner : inner), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
             const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int kKv, int kVL>
cudaError_t launch_d(const Params& p, cudaStream_t stream) {
  constexpr int kEsz = (kKv == kKvF16 || kKv == kKvBf16) ? 2 : 1;
  using S = Lay<D, kEsz, kKv == kKvBf16 ? 2 : 1>;
  CUtensorMap km, vm;
  const int64_t rows = (int64_t)p.num_pages * p.Hkv * p.bs;
  const int box_rows = p.bs < kT ? p.bs : kT;
  if (!encode_i8_map(&km, p.k_cache, rows, D, box_rows, kEsz)) return cudaErrorInvalidValue;
  // dimension-major V: [pages * Hkv * D rows][bs tokens], a box of box_rows tokens x D rows
  // (no map for 8-byte dim rows, which the kernel copies page by page)
  memset(&vm, 0, sizeof(vm));
  if (kVL != kVTok ? kVL == kVDim && !encode_i8_map(&vm, p.v_cache, (int64_t)p.num_pages * p.Hkv * D, p.bs, D, kEsz,
                                                box_rows)
           : !encode_i8_map(&vm, p.v_cache, rows, D, box_rows, kEsz))
    return cudaErrorInvalidValue;
  constexpr int smem = (int)S::kSmem;
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(&partial_tc_i8_kernel<D, kKv, kVL>), smem);
  if (e != cudaSuccess) return e;
  const int n_items = p.B * p.Hkv * p.num_splits;
  const int n_sm = sm_count();
  if (n_sm <= 0) return cudaErrorInvalidValue;
  dim3 grid(n_items < n_sm ? n_items : n_sm);
  partial_tc_i8_kernel<D, kKv, kVL><<<grid, kThreads, smem, stream>>>(p, km, vm);
  return cudaGetLastError();
}

template <int kKv, int kVL>
cudaError_t launch_kv(const Params& p, cudaStream_t stream) {
  switch (p.D) {
    case 64: return launch_d<64, kKv, kVL>(p, stream);
    case 128: return launch_d<128, kKv, kVL>(p, stream);
    case 256:
      // a 16-bit cache at head_dim 256: token-major V only (one-deep rings, batched widening)
      if constexpr (kKv == kKvI8 || kKv == kKvE4m3 || kVL == kVTok) return launch_d<256, kKv, kVL>(p, stream);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

template <int kKv>
cudaError_t launch_kv(const Params& p, cudaStream_t stream) {
  if (!p.v_dim_major) return launch_kv<kKv, kVTok>(p, stream);
  if constexpr (kKv == kKvI8 || kKv == kKvE4m3)
    if (p.bs < 16) return launch_kv<kKv, kVDim8>(p, stream);
  return launch_kv<kKv, kVDim>(p, stream);
}

}  // namespace

bool tc_i8_supports(const tllm_decode_attn_desc& d, int rows) {
  const int bs = d.block_size;
  const bool quant = d.kv_dtype == TLLM_INT8 || d.kv_dtype == TLLM_FP8_E4M3;
  const bool b16 = d.kv_dtype == TLLM_F16 || d.kv_dtype == TLLM_BF16;
  const bool v_ok = d.v_layout == TLLM_V_TOKEN_MAJOR || d.v_layout == TLLM_V_DIM_MAJOR;
  return (quant || b16) && (d.q_dtype == TLLM_BF16 || d.q_dtype == TLLM_F16) &&
         (d.head_dim == 64 || d.head_dim == 128 || (d.head_dim == 256 && (quant || d.v_layout == TLLM_V_TOKEN_MAJOR))) &&
         v_ok &&
         rows >= 1 && rows <= 128 && (bs == 8 || bs == 16 || bs == 32 || bs == 64 || bs == 128) &&
         (int64_t)d.num_pages * d.num_kv_heads * bs < ((int64_t)1 << 31) &&
         (int64_t)d.num_pages * d.num_kv_heads * d.head_dim < ((int64_t)1 << 31);   // (a transposed V's rows)
}

bool tc_i8_pointers_ok(const Params& p) {
  auto al = [](const void* x) { return ((uintptr_t)x & 15) == 0; };
  const bool quant = p.kv_dtype == TLLM_INT8 || p.kv_dtype == TLLM_FP8_E4M3;
  return al(p.q) && al(p.k_cache) && al(p.v_cache) && (!quant || (al(p.k_scales) && al(p.v_scales))) && al(p.out);
}

cudaError_t launch_partial_tc_i8(const Params& p, cudaStream_t stream) {
  switch (p.kv_dtype) {
    case TLLM_FP8_E4M3: return launch_kv<kKvE4m3>(p, stream);
    case TLLM_F16: return launch_kv<kKvF16>(p, stream);
    case TLLM_BF16: return launch_kv<kKvBf16>(p, stream);
    default: return launch_kv<kKvI8>(p, stream);
  }
}

}  // namespace tllm
