// FP8 tensor-core split-KV partial kernel for sm_103a: e4m3 KV with per-token fp32 K and V
// scales, head_dim 128, up to 64 packed rows (Hq/Hkv query heads x Lq query rows) per KV
// head, block size 8..128.
//
// Persistent CTAs, one per SM, take the real (request, kv head, split) items of a work list
// built on the device from the lengths, in turn (item k goes to CTA k mod grid, so a ragged
// batch spreads its items over all CTAs). Per item, each KV page of the split is read from HBM once
// (GQA packing: "split packed-Q8 verifier KV scans", hipfire PR #760, Summary). Roles:
//   warp 0      K producer: walks the block table (read one group of tiles ahead) and
//               TMA-loads each page's K slab (one 2-D box, 128-byte swizzle) into a 4-stage
//               K ring, released when the tile's QK^T is done;
//   warp 2      V producer: the same walk for the V slabs, into a 4-stage V ring released
//               when the tile's PV is done;
//   warp 1      one thread issues every QK^T (tcgen05.mma kind::f8f6f4, fp32 accumulators
//               in TMEM); warp 3: one thread issues every PV;
//   warps 4..7  softmax warpgroup 0: tiles 0, 2, 4, ...
//   warps 8..11 softmax warpgroup 1: tiles 1, 3, 5, ...
//               thread = (packed row, half of the 128-token tile). Each thread also fetches
//               the K / V scales of one token (its token duty) of the warpgroup's tile after
//               next (block-table entry, then the two scales, plain loads kept in registers
//               for a tile) into a 3-slot ring of the warpgroup, so no producer or barrier
//               stands between the scales and the softmax. Each warpgroup keeps its
//               own running (reference, sum, P scale) and its own S and O in TMEM (512 columns in
//               all); the two are merged once, in the epilogue. Two warps per SMSP hide each
//               other's TMEM-load, barrier and MUFU latencies.
//
// The contractions run on the FP8 tensor cores without converting the cache:
//   S = Q K^T: A = [Q_hi | Q_lo] along K (256 bytes per row), the 64 rows stored twice so
//              that M = 128; B = the K tile as loaded (K-major). Q (bf16: 8 significant
//              bits) is rescaled by a power of two and split into two e4m3 parts whose sum
//              represents it exactly except for elements far below the row maximum.
//   O += P V:  A = [P_hi ; P_lo] stacked on M (128 rows); B = the V tile as loaded
//              (MN-major). TMEM lanes 0..63 accumulate the hi part and 64..127 the lo part;
//              they are added once, in the epilogue.
// Softmax in log2 units (tiny-llm PR #11: per-split online (m, l, acc)); the K scale is
// folded into the score and the V scale into P, with a power-of-two factor 2^C that keeps
// P * vs inside the e4m3 range (C changes only when a larger V scale arrives; O is then
// rescaled exactly). The exponent reference of a row is its running maximum, moved only when
// a tile's maximum passes it by more than kSlack (any reference gives the same result once
// the sums are merged; a lagging one only makes P up to 2^kSlack), so O is rescaled on few
// tiles instead of whenever one of a warp's 32 rows sets a new maximum.
//
// Every wait is bounded in time; a timeout sets TLLM_FLAG_TIMEOUT, lets every role run to
// its end without waiting, drains the copies and MMAs in flight, skips the output stores,
// takes no further item and frees TMEM.
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace tllm {
namespace {

using namespace ptx;

constexpr int kTile = 128;      // tokens per tile
constexpr int kD = 128;         // head_dim
constexpr int kStages = 4;
constexpr int kSmThreads = 256;                  // one softmax warpgroup: 8 warps
constexpr int kThreads = 128 + 2 * kSmThreads;   // control warpgroup (2 producers, 2 MMA issuers) + 2 softmax
constexpr uint32_t kFull = 0xffffffffu;
constexpr int kCUnset = 1 << 20;
// Slack of the running row reference M (log2 units): M moves only when a tile's row maximum
// exceeds it by more than kSlack, so P = 2^(score - M) stays below 2^kSlack and the O rescale
// (a TMEM round trip) is rare; the P scale 2^C leaves room for that factor.
constexpr int kSlack = 2;

// shared-memory layout (byte offsets from a 1024-aligned base)
// K tiles (released when the tile's QK^T is done), V tiles (released when its PV is done) and
// per warpgroup a 3-slot ring of per-token scales and token masks (written and read by the
// warpgroup itself).
constexpr int kScSlots = 3;
constexpr uint32_t kKStageBytes = 16384, kVStageBytes = 16384;
// meta: 4 token-mask words, then the V-scale maximum of each of the 4 duty warps' 32 tokens
constexpr uint32_t kScKs = 0, kScVs = 512, kScMeta = 1024, kScVmax = 1040, kScStageBytes = 1056;
constexpr uint32_t kOffV = kStages * kKStageBytes;
constexpr uint32_t kOffA = kOffV + kStages * kVStageBytes;   // Q hi | Q lo, 2 x 16 KB
constexpr uint32_t kOffP = kOffA + 32768;                    // P of warpgroup 0 | 1, 2 x 16 KB
constexpr uint32_t kOffSc = kOffP + 32768;                   // scale ring
constexpr uint32_t kOffX = kOffSc + 2 * kScSlots * kScStageBytes;  // exchange floats
constexpr int kXSlot = 264, kXL = 2 * kXSlot;                // exchange: 2 tile slots, then row sums
constexpr uint32_t kXWg = 4096;                              // bytes per warpgroup (784 floats used)
constexpr uint32_t kOffJoint = kOffX + 2 * kXWg;
constexpr uint32_t kOffBar = kOffJoint + 1280;
constexpr uint32_t kNumBars = 4 * kStages + 2 + 2 + 2 + 2 + 2 + 2;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kOffList = kOffMisc + 64;                 // work list + its scan scratch
constexpr uint32_t kSmemBytes = kOffList + kListWords * 4 + 1024;   // + alignment slack
static_assert(kOffV % 1024 == 0 && kOffA % 1024 == 0, "stage alignment");
static_assert(2 * 64 * 128 * 4 <= kStages * (kKStageBytes + kVStageBytes), "epilogue exchange B: K + V rings");
static_assert(64 * 128 * 4 <= 32768, "epilogue exchange C: the Q area");
static_assert(kSmemBytes <= 232448, "shared memory");

// TMEM columns: S of warpgroup w at 128 w, O of warpgroup w at 256 + 128 w
constexpr uint32_t kTmemCols = 512, kColS = 0, kColO = 256;

// byte offset of (row, byte) inside a [rows][128 B] tile in the 128-byte swizzle layout
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t byte) {
  return (row >> 3) * 1024 + (row & 7) * 128 + ((((byte >> 4) ^ row) & 7) << 4) + (byte & 15);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }   // e in [-126, 127]

// mbarriers (8 bytes each, from kOffBar), named by their shared-memory address
constexpr uint32_t kBarKFull = 0, kBarKEmpty = kStages, kBarVFull = 2 * kStages, kBarVEmpty = 3 * kStages,
                   kBarSFull = 4 * kStages, kBarSFree = kBarSFull + 2, kBarPFull = kBarSFree + 2, kBarPvDone = kBarPFull + 2,
                   kBarQFull = kBarPvDone + 2, kBarMmaFin = kBarQFull + 1, kBarXMax = kBarMmaFin + 1;
static_assert(kBarXMax + 2 == kNumBars, "barrier count");
struct Bars {
  uint32_t base;
  __device__ uint32_t at(uint32_t i) const { return base + 8u * i; }
  __device__ uint32_t k_full(int s) const { return at(kBarKFull + s); }      // K producer -> MMA (tx bytes)
  __device__ uint32_t k_empty(int s) const { return at(kBarKEmpty + s); }    // MMA commit after QK^T
  __device__ uint32_t v_full(int s) const { return at(kBarVFull + s); }      // V producer -> MMA (tx bytes)
  __device__ uint32_t v_empty(int s) const { return at(kBarVEmpty + s); }    // MMA commit after PV
  __device__ uint32_t s_full(int w) const { return at(kBarSFull + w); }      // QK^T of a tile done (buffer = warpgroup)
  __device__ uint32_t s_free(int w) const { return at(kBarSFree + w); }      // S read out of TMEM
  __device__ uint32_t p_full(int w) const { return at(kBarPFull + w); }      // P written, O rescaled
  __device__ uint32_t pv_done(int w) const { return at(kBarPvDone + w); }    // PV of a tile done
  __device__ uint32_t q_full() const { return at(kBarQFull); }               // Q in shared memory
  __device__ uint32_t mma_fin() const { return at(kBarMmaFin); }             // final commits of the two MMA issuers
  __device__ uint32_t x_max(int w) const { return at(kBarXMax + w); }        // row partial maxima of a tile written
};

// abort: shared-memory address of the CTA's abort word
__device__ __forceinline__ void set_abort(uint32_t abort, uint32_t* status) {
  if (!ld_volatile_shared(abort)) {
    asm volatile("st.volatile.shared.b32 [%0], %1;" ::"r"(abort), "r"(1) : "memory");
    atomicOr(status, TLLM_FLAG_TIMEOUT);
  }
}

// kVdm: the V cache is dimension-major ([pages, Hkv, D, bs]); a separate instance, so the
// token-major one is compiled exactly as without it
template <bool kVdm>
__global__ void __launch_bounds__(kThreads)
    partial_tc_fp8_kernel(const Params p, const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) pdl_launch_dependents();
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffMisc);
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  int* wlist = reinterpret_cast<int*>(sm + kOffList);

  // Persistent: the CTAs (one per SM at most) take the real (request x kv head, split) items of
  // the work list in turn. Each item runs its own pipeline from scratch (barriers re-initialised
  // once the previous item has drained).
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
  const int n_tiles = t1 > t0 ? (t1 - t0 + kTile - 1) / kTile : 0;
  const bool finalize = sp.nsplit == 1;
  const int u_split = u * p.max_splits + split;

  if (n_tiles == 0) {                      // nothing visible: zero rows
    for (int idx = tid; idx < p.R * kD; idx += kThreads) {
      const int r = idx / kD, d = idx % kD;
      if (finalize) {
        const int i = r / p.G, hq = g * p.G + r % p.G;
        store_f32(p.out, p.out_dtype, ((int64_t)(b * p.Lq + i) * p.Hq + hq) * kD + d, 0.f);
      } else {
        store_rec(p, ((int64_t)u_split * p.R + r) * kD + d, 0.f);
        if (d == 0) p.ws_lse[(int64_t)u_split * p.R + r] = -INFINITY;
      }
    }
    continue;
  }

  const int bs = p.bs;
  // bs is a power of two (8..128): block-size arithmetic uses shifts and masks
  const int bs_sh = __ffs(bs) - 1;
  const int ppt_sh = 7 - bs_sh;                      // log2(pages per tile)
  const int ppt = 1 << ppt_sh;                       // pages per tile (1..16)
  const int gt_sh = 5 - ppt_sh, gt = 1 << gt_sh;     // a producer's page-id group: 32 / ppt tiles
  // Page ids of the producers are read one group of tiles ahead (one entry per lane), so
  // the block-table latency stays off the refill path.
  auto fetch = [&](int grp, int& pg, int& need) {
    const int tile = (grp << gt_sh) + (lane >> ppt_sh), slot = lane & (ppt - 1);
    pg = 0;
    need = 0;
    if (tile < n_tiles) {
      const int tt = t0 + tile * kTile, first = tt + slot * bs;
      if (max(first, sp.lo) < min(first + bs, t1)) {
        need = 1;
        pg = page_at(p, b, (tt >> bs_sh) + slot);
      }
    }
  };
  // Start-up loads go out before the set-up barrier so that their latencies overlap: the
  // producers' first two page-id groups and tensor maps, warpgroup 0's query rows.
  int pg_cur = 0, nd_cur = 0, pg_nxt = 0, nd_nxt = 0;
  if (warp == 0 || warp == 2) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(warp == 0 ? &kmap : &vmap)) : "memory");
    fetch(0, pg_cur, nd_cur);
    fetch(1, pg_nxt, nd_nxt);
  }
  // the first 64 bytes of this thread's 32 query elements (all of them for a 16-bit Q)
  uint4 qraw[4] = {};
  const uint4* qsrc = nullptr;
  if (warp >= 4 && warp < 12) {
    const int L0 = 32 * (warp & 3) + lane, r0 = L0 & 63;
    const int tok00 = 64 * (L0 >> 6) + 32 * (((warp - 4) & 7) >> 2);
    if (r0 < p.R) {
      const int qi0 = r0 / p.G, qh0 = g * p.G + r0 % p.G;
      const int64_t e0 = ((int64_t)(b * p.Lq + qi0) * p.Hq + qh0) * kD + tok00;
      qsrc = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.q) + e0 * (p.q_dtype == TLLM_F32 ? 4 : 2));
#pragma unroll
      for (int c = 0; c < 4; c++) qraw[c] = __ldg(qsrc + c);
    }
  }

  const Bars bars{sbase + kOffBar};
  const uint32_t abort = sbase + kOffMisc + 4;
  int* qexp_slot = reinterpret_cast<int*>(sm + kOffMisc + 8);

  if (tid == 0) {
    for (int s = 0; s < kStages; s++) {
      mbar_init(bars.k_full(s), 1);
      mbar_init(bars.k_empty(s), 1);
      mbar_init(bars.v_full(s), 1);
      mbar_init(bars.v_empty(s), 1);
    }
    for (int s = 0; s < 2; s++) {
      mbar_init(bars.s_full(s), 1);
      mbar_init(bars.s_free(s), kSmThreads / 32);   // one elected lane per softmax warp
      mbar_init(bars.p_full(s), kSmThreads / 32);
      mbar_init(bars.pv_done(s), 1);
    }
    mbar_init(bars.q_full(), kSmThreads / 32);
    mbar_init(bars.x_max(0), kSmThreads / 32);
    mbar_init(bars.x_max(1), kSmThreads / 32);
    mbar_init(bars.mma_fin(), 2);
    *reinterpret_cast<volatile int*>(sm + kOffMisc + 4) = 0;
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp < 4) {
   if (warp == 0 || warp == 2) {
    // ---------------- producers: warp 0 K tiles, warp 2 V tiles ----------------
    const bool isk = warp == 0;
    const uint32_t full = isk ? bars.k_full(0) : bars.v_full(0);
    const uint32_t empty = isk ? bars.k_empty(0) : bars.v_empty(0);
    // Two tiles per iteration: lanes [0, ppt) serve tile j0 and lanes [ppt, 2 ppt) tile j0 + 1,
    // so the warp's short dependent chain (page lookup, ballot, expect_tx, TMA) is paid once
    // per two tiles. A group holds an even number of tiles, so a pair never straddles groups.
    int issued = 0;
    for (int j0 = 0; j0 < n_tiles; j0 += 2) {
      if (j0 > 0 && (j0 & (gt - 1)) == 0) {
        pg_cur = pg_nxt;
        nd_cur = nd_nxt;
        fetch((j0 >> gt_sh) + 1, pg_nxt, nd_nxt);
      }
      const int ntl = min(2, n_tiles - j0);          // tiles in this iteration
      for (int d = 0; d < ntl; d++) {
        const int j = j0 + d;
        if (j >= kStages && !mbar_wait(empty + 8 * (j % kStages), ((j / kStages) - 1) & 1, abort))
          set_abort(abort, p.status);
      }
      if (ld_volatile_shared(abort)) break;
      const int src = (((j0 & (gt - 1)) << ppt_sh) + lane) & 31;
      const int pgv = __shfl_sync(kFull, pg_cur, src);
      const int ndv = __shfl_sync(kFull, nd_cur, src);
      const int dl = lane >> ppt_sh, slot = lane & (ppt - 1);  // this lane's tile of the pair and page slot
      const int jl = j0 + dl;
      int page = -1;
      if (dl < ntl && ndv) {
        if (pgv < 0 || pgv >= p.num_pages) {
          if (isk) atomicOr(p.status, TLLM_FLAG_BAD_PAGE);
        } else {
          page = pgv;
        }
      }
      const uint32_t pair_mask = __ballot_sync(kFull, page >= 0);
      const uint32_t tmask = ppt >= 32 ? kFull : ((1u << ppt) - 1u);
      if (slot == 0 && dl < ntl) {
        const uint32_t m = (pair_mask >> (dl * ppt)) & tmask;
        mbar_arrive_expect_tx(full + 8 * (jl % kStages), __popc(m) * (uint32_t)bs * kD);
      }
      __syncwarp();
      if (page >= 0) {
        const int64_t row = ((int64_t)page * p.Hkv + g) * bs;
        const int st = jl % kStages;
        if (isk) {
          tma_load_2d(sbase + st * kKStageBytes + slot * bs * kD, &kmap, 0, (int)row, full + 8 * (st));
        } else if constexpr (!kVdm) {
          tma_load_2d(sbase + kOffV + st * kVStageBytes + slot * bs * kD, &vmap, 0, (int)row, full + 8 * (st));
        } else {
          // dimension-major V page: bs / 16 boxes of 128 dims x 16 tokens, each a 2 KB block of
          // core matrices; block k of the tile holds its tokens 16 k .. 16 k + 15
          for (int c = 0; c < (bs >> 4); c++)
            tma_load_2d(sbase + kOffV + st * kVStageBytes + (slot * (bs >> 4) + c) * 2048u, &vmap, 16 * c,
                        (int)(row / bs * kD), full + 8 * (st));
        }
      }
      issued = j0 + ntl;
    }
    // drain: every issued stage's copies must land before the CTA can exit
    for (int j = max(0, issued - kStages); j < issued; j++)
      if (!mbar_wait(full + 8 * (j % kStages), (j / kStages) & 1, 0u)) set_abort(abort, p.status);
    // ... and the release of each of those stages by its MMA (an asynchronous tcgen05.commit
    // arrival) must have landed too, before the next item re-initialises the barriers
    for (int j = max(0, issued - kStages); j < issued; j++)
      if (!mbar_wait(empty + 8 * (j % kStages), (j / kStages) & 1, abort)) set_abort(abort, p.status);
   } else if (lane == 0) {
    // ---------------- MMA issuers: warp 1 issues every QK^T, warp 3 every PV ----------------
    // Each thread blocks only on its own inputs; tcgen05.commit tracks the committing
    // thread's own MMAs, so the two streams stay independent.
    bool ok = true;
    if (warp == 1) {
      const uint32_t idqk = idesc_e4m3(128, 128, 0, 0);
      const uint32_t a0 = sbase + kOffA, a1 = sbase + kOffA + 16384;
      ok = mbar_wait(bars.q_full(), 0, abort);
      for (int j = 0; ok && j < n_tiles; j++) {
        const int st = j % kStages, sb = j & 1;
        if (!mbar_wait(bars.k_full(st), (j / kStages) & 1, abort)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(bars.s_free(sb), ((j >> 1) - 1) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kt = sbase + st * kKStageBytes;
#pragma unroll
        for (int k = 0; k < 8; k++) {
          const uint32_t a = (k < 4 ? a0 : a1) + 32 * (k & 3);
          mma_e4m3(tmem + kColS + sb * 128, sdesc_sw128(a, 16, 1024), sdesc_sw128(kt + 32 * (k & 3), 16, 1024),
                   idqk, k > 0 ? 1u : 0u);
        }
        mma_commit(bars.s_full(sb));
        mma_commit(bars.k_empty(st));
      }
    } else {
      // V as loaded: token-major pages give an MN-major B (dims contiguous, 128-byte swizzle);
      // dimension-major pages a K-major B of 16-token core-matrix blocks, 2 KB apart along K
      const uint32_t idpv = idesc_e4m3(128, 128, 0, kVdm ? 0 : 1);
      for (int j = 0; ok && j < n_tiles; j++) {
        const int pb = j & 1, st = j % kStages;
        if (!mbar_wait(bars.p_full(pb), (j >> 1) & 1, abort)) { ok = false; break; }
        if (!mbar_wait(bars.v_full(st), (j / kStages) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t vt = sbase + kOffV + st * kVStageBytes;
        const uint32_t pa = sbase + kOffP + pb * 16384;
#pragma unroll
        for (int k = 0; k < 4; k++)
          mma_e4m3(tmem + kColO + pb * 128, sdesc_sw128(pa + 32 * k, 16, 1024),
                   kVdm ? sdesc_none(vt + 4096 * k, 2048, 128) : sdesc_sw128(vt + 4096 * k, 16384, 1024), idpv,
                   (j >= 2 || k > 0) ? 1u : 0u);
        mma_commit(bars.pv_done(pb));
        mma_commit(bars.v_empty(st));
      }
    }
    if (!ok) set_abort(abort, p.status);
    // every MMA issued must finish before TMEM is released (both issuers commit here)
    mma_commit(bars.mma_fin());
    if (!mbar_wait(bars.mma_fin(), 0, 0u)) set_abort(abort, p.status);
   }
   // lanes 1..31 of the issuer warps wait here for their lane 0, so that every warp reaches the
   // item's closing CTA barrier (an aligned barrier) converged
   if (warp == 1 || warp == 3) __syncwarp();
  } else {
    // ---------------- softmax warpgroups: 8 warps each; warpgroup w takes tiles w, w + 2, ... ----------------
    // Thread = (TMEM lane L = packed row r and token half h, column part c): it owns the 32
    // tokens tok0 .. tok0 + 31 of every tile of its warpgroup and, in O, the 64 columns of part c.
    const int wg = (warp - 4) >> 3;
    const int sub = (warp - 4) & 7;
    const int wq = warp & 3;                      // TMEM lane quadrant of this warp
    const int cpart = sub >> 2;                   // column part (0 or 1)
    const int L = 32 * wq + lane;                 // TMEM lane = A / P / O row
    const int r = L & 63, h = L >> 6;             // packed row, token half
    const int tok0 = 64 * h + 32 * cpart;         // first token of this thread inside a tile
    const int xq = 2 * h + cpart;                 // which of the row's 4 partials this thread holds
    const bool duty = cpart == 0;                 // part-0 warps fetch the scales: token kt each
    const int kt = L;                             // token duty inside a tile (0..127)
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    const uint32_t bar_id = 1 + wg;               // 256 threads
    // per-warpgroup exchange: [slot][0,256) row maxima (partial xq at 64 xq + r; slot = tile
    // parity), then [kXL, kXL + 256) row sums
    float* xw = reinterpret_cast<float*>(sm + kOffX + wg * kXWg);
    float* xj = reinterpret_cast<float*>(sm + kOffJoint);   // [0,128) M_w, [128,256) l_w, [256,258) C_w

    const bool real = r < p.R;
    const int qi = real ? r / p.G : 0;
    const int qh = g * p.G + (real ? r % p.G : 0);
    // (the scale ring is fed before Q is ready: it does not depend on Q)
    // Token duty kt of tile jt: its page (rd = false if the token is not read by this split)
    // and its two scales (ok = false if it is not read or its page id is out of range). The
    // loads are unconditional, at a clamped in-bounds address (token 0 / page 0), so nothing
    // waits for them until their values are stored, one tile later; put() applies ok.
    auto tok_page = [&](int jt, int& pg) -> bool {
      const int t = t0 + jt * kTile + kt;
      const bool rd = jt < n_tiles && t >= sp.lo && t < t1;
      pg = page_at(p, b, rd ? t >> bs_sh : 0);
      return rd;
    };
    auto tok_scales = [&](int jt, bool rd, int pg, float& ks, float& vs) -> bool {
      const bool ok = rd && pg >= 0 && pg < p.num_pages;
      const int64_t a = ((int64_t)(ok ? pg : 0) * p.Hkv + g) * bs + ((t0 + jt * kTile + kt) & (bs - 1));
      ks = __ldg(p.k_scales + a);
      vs = __ldg(p.v_scales + a);
      return ok;
    };
    auto ring = [&](int jt) -> uint8_t* {
      return sm + kOffSc + (wg * kScSlots + (jt >> 1) % kScSlots) * kScStageBytes;
    };
    auto put = [&](int jt, float ks, float vs, bool ok) {
      uint8_t* sl = ring(jt);
      reinterpret_cast<float*>(sl + kScKs)[kt] = ok ? ks : 0.f;
      reinterpret_cast<float*>(sl + kScVs)[kt] = ok ? vs : 0.f;
      const uint32_t m = __ballot_sync(kFull, ok);
      const float vm = warp_max_abs(ok ? vs : 0.f);
      if (lane == 0) {
        reinterpret_cast<uint32_t*>(sl + kScMeta)[wq] = m;
        reinterpret_cast<float*>(sl + kScVmax)[wq] = vm;
      }
    };
    // pipeline (duty warps): tile wg in the ring, tile wg + 2 in registers, the page of tile
    // wg + 4 in flight
    int pgC = 0;
    bool rdC = false, okA = false, okB = false;
    float ksA = 0.f, vsA = 0.f, ksB = 0.f, vsB = 0.f;
    if (duty) {
      int pgA, pgB;
      const bool rdA = tok_page(wg, pgA), rdB = tok_page(wg + 2, pgB);
      rdC = tok_page(wg + 4, pgC);
      okA = tok_scales(wg, rdA, pgA, ksA, vsA);
      okB = tok_scales(wg + 2, rdB, pgB, ksB, vsB);
      put(wg, ksA, vsA, okA);
    }
    named_bar(bar_id, kSmThreads);

    int qexp = 0;                                 // Q scale exponent (same value in every thread)
    if (wg == 0) {
      // Q rows -> e4m3 hi/lo, CTA-wide power-of-two scale; this thread converts 32 dims.
      // (loaded at kernel start: qraw; an fp32 Q has its second 64 bytes fetched now)
      float qv[32];
      {
        VecF32<32> v;
#pragma unroll
        for (int c = 0; c < 4; c++) v.raw[c] = qraw[c];
#pragma unroll
        for (int c = 4; c < 8; c++)
          v.raw[c] = (qsrc && p.q_dtype == TLLM_F32) ? __ldg(qsrc + c) : make_uint4(0, 0, 0, 0);
        v.get(p.q_dtype, qv);
      }
      float amax = 0.f;
#pragma unroll
      for (int d = 0; d < 32; d++) amax = fmaxf(amax, fabsf(qv[d]));
      amax = warp_max_abs(amax);
      if (lane == 0) xj[260 + sub] = amax;
      named_bar(bar_id, kSmThreads);
      const float4 a0 = *reinterpret_cast<const float4*>(xj + 260), a1 = *reinterpret_cast<const float4*>(xj + 264);
      amax = fmaxf(fmaxf(fmaxf(a0.x, a0.y), fmaxf(a0.z, a0.w)), fmaxf(fmaxf(a1.x, a1.y), fmaxf(a1.z, a1.w)));
      if (amax > 0.f) {
        int ex;
        frexpf(amax, &ex);
        qexp = 8 - ex;                            // amax * 2^qexp in [128, 256)
      }
      const float qmul = ldexpf(1.f, qexp);
#pragma unroll
      for (int cc = 0; cc < 2; cc++) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int w = 0; w < 4; w++) {
          uint32_t hb = 0, lb = 0;
#pragma unroll
          for (int pr = 0; pr < 2; pr++) {
            const int d = 16 * cc + 4 * w + 2 * pr;
            const float x0 = qv[d] * qmul, x1 = qv[d + 1] * qmul;
            const uint16_t hi = f32x2_to_e4m3x2(x1, x0);
            const float2 hf = f16x2_to_f32x2(e4m3x2_to_f16x2(hi));
            const uint16_t lo = f32x2_to_e4m3x2(x1 - hf.y, x0 - hf.x);
            hb |= (uint32_t)hi << (16 * pr);
            lb |= (uint32_t)lo << (16 * pr);
          }
          hw[w] = hb;
          lw[w] = lb;
        }
        const uint32_t byte = tok0 + 16 * cc;
        for (int dup = 0; dup < 2; dup++) {
          const uint32_t row = r + 64 * dup;
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sbase + kOffA + sw128(row, byte)),
                       "r"(hw[0]), "r"(hw[1]), "r"(hw[2]), "r"(hw[3]));
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sbase + kOffA + 16384 + sw128(row, byte)),
                       "r"(lw[0]), "r"(lw[1]), "r"(lw[2]), "r"(lw[3]));
        }
      }
      if (tid == 128) *qexp_slot = qexp;
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.q_full());
    }
    if (wg == 1) {
      // warpgroup 1 reads the exponent once q_full (which the writer's warp arrives on after
      // the store) completes
      if (!mbar_wait(bars.q_full(), 0, abort)) set_abort(abort, p.status);
      qexp = *reinterpret_cast<volatile int*>(qexp_slot);
    }
    const float qscale = p.scale_log2 * ldexpf(1.f, -qexp);

    const int pos = real ? ctx - p.Lq + qi : -1;   // position of the row
    const int pos_lo = ctx - p.Lq;                  // lowest real row position

    float M = -INFINITY, l = 0.f;                   // l: this thread's partial row sum, units of 2^-C
    int C = kCUnset;
    int last = -1;
    for (int j = wg; j < n_tiles; j += 2) {
      last = j;
      const int st = j % kStages;
      const int tt = t0 + j * kTile;
      // this thread's 32 scores out of TMEM: the load runs while the scale ring is fed
      if (!mbar_wait(bars.s_full(wg), (j >> 1) & 1, abort)) set_abort(abort, p.status);
      tc_fence_after();
      uint32_t sreg[32];
      tmem_ld32(tmem + lane_off + kColS + wg * 128 + tok0, sreg);
      if (duty) {
        // tile j + 2's scales into the ring (published to the warpgroup by this tile's
        // row-maximum barrier, which every warp arrives on after this store), then the next fetches
        put(j + 2, ksB, vsB, okB);
        okB = tok_scales(j + 4, rdC, pgC, ksB, vsB);
        rdC = tok_page(j + 6, pgC);
      }
      const uint8_t* stp = ring(j);
      float* xs = xw + kXSlot * ((j >> 1) & 1);
      const uint4 vmk = *reinterpret_cast<const uint4*>(stp + kScMeta);   // token mask of the tile
      const bool partial = (vmk.x & vmk.y & vmk.z & vmk.w) != kFull;
      if (partial && duty) {
        // Tokens this split does not read (their scales are already zero): their V rows become
        // zero too, so stale or poisoned bytes never reach an MMA. The p_full arrival below
        // (after a proxy fence) publishes the zeros to the PV MMA.
        if (!mbar_wait(bars.v_full(st), (j / kStages) & 1, abort)) set_abort(abort, p.status);
        const uint32_t mw = wq == 0 ? vmk.x : wq == 1 ? vmk.y : wq == 2 ? vmk.z : vmk.w;
        if (!((mw >> lane) & 1)) {
          if constexpr (!kVdm) {
            const uint32_t vrow = sbase + kOffV + st * kVStageBytes + 128 * kt;
#pragma unroll
            for (int c = 0; c < 8; c++)
              asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(vrow + 16 * c), "r"(0));
          } else {
            // the token's byte in each of the 128 dimension rows of its 16-token block
            const uint32_t vcol = sbase + kOffV + st * kVStageBytes + (kt >> 4) * 2048u + (kt & 15);
            for (int d = 0; d < kD; d++) asm volatile("st.shared.u8 [%0], %1;" ::"r"(vcol + 16 * d), "h"((uint16_t)0));
          }
        }
        fence_proxy_async();
      }
      const bool masked = partial || tt + kTile - 1 > pos_lo || (p.window > 0 && tt < ctx - p.window);

      tmem_ld_wait(sreg);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.s_free(wg));

      const float4* ks4 = reinterpret_cast<const float4*>(stp + kScKs) + tok0 / 4;
      const float4* vs4 = reinterpret_cast<const float4*>(stp + kScVs) + tok0 / 4;
      // u = raw score x K scale; the score in log2 units is u * qscale (qscale > 0)
      float u[32];
      if (!masked) {
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
        const float* ks = reinterpret_cast<const float*>(ks4);
        const uint32_t vw = xq == 0 ? vmk.x : xq == 1 ? vmk.y : xq == 2 ? vmk.z : vmk.w;
#pragma unroll
        for (int i = 0; i < 32; i++) {
          const int t = tt + tok0 + i;
          const bool vis = ((vw >> i) & 1) && t <= pos && (p.window <= 0 || pos - t < p.window);
          u[i] = vis ? __uint_as_float(sreg[i]) * ks[i] : -INFINITY;
        }
      }
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int k = 0; k < 16; k++) m4[k & 3] = fmax3(m4[k & 3], u[2 * k], u[2 * k + 1]);
      const float mloc = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
      // Split-phase exchange of the row maximum: this thread's partial is published now, P is
      // computed against a provisional reference, and the other three partials of the row are
      // waited for only before P is corrected and stored.
      xs[64 * xq + r] = mloc;
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.x_max(wg));

      // P scale exponent C from the tile's V-scale maximum (stored in the ring with the scales):
      // vmax * 2^C < 2^(8 - kSlack), so P * vs * 2^C < 256 while P stays below 2^kSlack; C only
      // ever decreases (then O is rescaled)
      const float4 vm4 = *reinterpret_cast<const float4*>(stp + kScVmax);
      const float vmax = fmaxf(fmaxf(vm4.x, vm4.y), fmaxf(vm4.z, vm4.w));
      int cdelta = 0;
      if (vmax > 0.f) {
        const int c = min(60, max(-60, 8 - kSlack - exponent_of(vmax)));
        if (C == kCUnset) C = c;
        else if (c < C) { cdelta = c - C; C = c; }
      } else if (C == kCUnset) {
        C = 0;
      }
      // Provisional reference: the row's, or this thread's own maximum when that passes it by
      // more than kSlack (P <= 2^C then). Either way P stays in range, and once the row's maximum
      // is known P is multiplied by 2^(Rt - M_new) <= 1.
      const float ml2 = mloc * qscale;
      const float Rt = ml2 > M + (float)kSlack ? ml2 : M;
      const float e0 = Rt == -INFINITY ? 0.f : (float)C - Rt;   // p' = 2^(u qscale - Rt + C)
      const float2 qs2 = make_float2(qscale, qscale), e02 = make_float2(e0, e0);
      float2 ls = make_float2(0.f, 0.f);
#pragma unroll
      for (int i4 = 0; i4 < 8; i4++) {
        const float4 v = vs4[i4];                 // zero for tokens this split does not read
        const float2 x01 = ffma2(make_float2(u[4 * i4], u[4 * i4 + 1]), qs2, e02);
        const float2 x23 = ffma2(make_float2(u[4 * i4 + 2], u[4 * i4 + 3]), qs2, e02);
        const float2 p01 = make_float2(ex2(x01.x), ex2(x01.y)), p23 = make_float2(ex2(x23.x), ex2(x23.y));
        ls = fadd2(ls, fadd2(p01, p23));
        const float2 w01 = fmul2(p01, make_float2(v.x, v.y)), w23 = fmul2(p23, make_float2(v.z, v.w));
        u[4 * i4] = w01.x;                        // u now holds P * vs * 2^C against Rt
        u[4 * i4 + 1] = w01.y;
        u[4 * i4 + 2] = w23.x;
        u[4 * i4 + 3] = w23.y;
      }

      if (!mbar_wait(bars.x_max(wg), (j >> 1) & 1, abort)) set_abort(abort, p.status);
      const float mx = fmaxf(fmaxf(xs[r], xs[64 + r]), fmaxf(xs[128 + r], xs[192 + r])) * qscale;
      // the row reference moves only when the tile's maximum passes it by more than kSlack
      const float M_new = mx > M + (float)kSlack ? mx : M;
      const float fix = (Rt == M_new || Rt == -INFINITY) ? 1.f : ex2(Rt - M_new);
      const float alpha = M_new == -INFINITY ? 1.f : ex2(M - M_new);
      const float factor = alpha * pow2i(cdelta);
      if (__any_sync(kFull, fix != 1.f)) {
        const float2 f2 = make_float2(fix, fix);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 x = fmul2(make_float2(u[i], u[i + 1]), f2);
          u[i] = x.x;
          u[i + 1] = x.y;
        }
      }
      uint32_t hw[8], lw[8];
#pragma unroll
      for (int i4 = 0; i4 < 8; i4++)
        f16x4_split_e4m3(f32x2_to_f16x2(u[4 * i4 + 1], u[4 * i4]), f32x2_to_f16x2(u[4 * i4 + 3], u[4 * i4 + 2]),
                         hw[i4], lw[i4]);
      l = l * factor + (ls.x + ls.y) * fix;
      const float prev_M = M;
      M = M_new;

      // this warpgroup's P buffer and O are free once its previous PV (tile j - 2) is done
      if (j >= 2 && !mbar_wait(bars.pv_done(wg), ((j - 2) >> 1) & 1, abort)) set_abort(abort, p.status);
      const uint32_t pbase = sbase + kOffP + wg * 16384;
#pragma unroll
      for (int cc = 0; cc < 2; cc++) {
        const uint32_t byte = tok0 + 16 * cc;
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(pbase + sw128(r, byte)), "r"(hw[4 * cc]),
                     "r"(hw[4 * cc + 1]), "r"(hw[4 * cc + 2]), "r"(hw[4 * cc + 3]));
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(pbase + sw128(64 + r, byte)), "r"(lw[4 * cc]),
                     "r"(lw[4 * cc + 1]), "r"(lw[4 * cc + 2]), "r"(lw[4 * cc + 3]));
      }
      fence_proxy_async();

      // rescale O (this thread: lane L, the 64 columns of part c) when the row reference moved or
      // the P scale shrank (O holds this warpgroup's tiles < j)
      const bool need = j >= 2 && factor != 1.f && prev_M != -INFINITY;
      if (__any_sync(kFull, need)) {
        tc_fence_after();
        const float f = need ? factor : 1.f;
        const float2 f2 = make_float2(f, f);
        uint32_t o[64];
        tmem_ld64(tmem + lane_off + kColO + wg * 128 + 64 * cpart, o);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const float2 x = fmul2(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), f2);
          o[i] = __float_as_uint(x.x);
          o[i + 1] = __float_as_uint(x.y);
        }
        tmem_st64(tmem + lane_off + kColO + wg * 128 + 64 * cpart, o);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.p_full(wg));
    }

    // ---------------- epilogue: merge the two warpgroups' (M, l, O) ----------------
    if (last >= 0 && !mbar_wait(bars.pv_done(wg), (last >> 1) & 1, abort)) set_abort(abort, p.status);
    tc_fence_after();
    xw[kXL + 64 * xq + r] = l;
    named_bar(bar_id, kSmThreads);
    const float lw_tot = (xw[kXL + r] + xw[kXL + 64 + r]) + (xw[kXL + 128 + r] + xw[kXL + 192 + r]);
    if (xq == 0) {
      xj[64 * wg + r] = M;
      xj[128 + 64 * wg + r] = lw_tot;
      if (r == 0) xj[256 + wg] = C == kCUnset ? 0.f : (float)C;
    }
    named_bar(3, 2 * kSmThreads);
    const float M0 = xj[r], M1 = xj[64 + r];
    const float Mx = fmaxf(M0, M1);
    const float g0 = M0 == -INFINITY ? 0.f : ex2(M0 - xj[256] - Mx);
    const float g1 = M1 == -INFINITY ? 0.f : ex2(M1 - xj[257] - Mx);
    const float den = g0 * xj[128 + r] + g1 * xj[192 + r];
    // Exchange rows of 128 floats, float4 chunk c of row x stored at chunk c ^ (x & 7)
    // (conflict-free for 8 consecutive rows): xB = [L] in the K ring, xC = [r] in the Q area.
    float* xB = reinterpret_cast<float*>(sm);
    float* xC = reinterpret_cast<float*>(sm + kOffA);
    auto chunk = [](float* base, int row, int c4) -> float4* {
      return reinterpret_cast<float4*>(base + row * 128 + ((c4 ^ (row & 7)) << 2));
    };
    const int col0 = 64 * cpart;                    // this thread's O columns: col0 .. col0 + 63
    if (wg == 1) {
      uint32_t o[64];
      tmem_ld64(tmem + lane_off + kColO + 128 + col0, o);
      tmem_ld_wait();
#pragma unroll
      for (int i4 = 0; i4 < 16; i4++)
        *chunk(xB, L, col0 / 4 + i4) =
            last >= 0 ? make_float4(__uint_as_float(o[4 * i4]) * g1, __uint_as_float(o[4 * i4 + 1]) * g1,
                                    __uint_as_float(o[4 * i4 + 2]) * g1, __uint_as_float(o[4 * i4 + 3]) * g1)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    named_bar(3, 2 * kSmThreads);
    if (wg == 0) {
      // lane L holds part h (hi or lo) of row r: h = 0 keeps columns col0 .. col0 + 31 and sends
      // col0 + 32 .. col0 + 63 to the h = 1 thread of the row, which keeps the other 32
      const int c_send = col0 + 32 * (1 - h), c_keep = col0 + 32 * h;
      uint32_t o[32];
      tmem_ld32(tmem + lane_off + kColO + c_send, o);
      tmem_ld_wait();
#pragma unroll
      for (int i4 = 0; i4 < 8; i4++) {
        const float4 x = *chunk(xB, L, c_send / 4 + i4);
        *chunk(xC, r, c_send / 4 + i4) =
            make_float4(__uint_as_float(o[4 * i4]) * g0 + x.x, __uint_as_float(o[4 * i4 + 1]) * g0 + x.y,
                        __uint_as_float(o[4 * i4 + 2]) * g0 + x.z, __uint_as_float(o[4 * i4 + 3]) * g0 + x.w);
      }
      tmem_ld32(tmem + lane_off + kColO + c_keep, o);
      tmem_ld_wait();
      named_bar(bar_id, kSmThreads);
      if (real && !ld_volatile_shared(abort)) {
        float mul = 0.f;
        if (finalize) {
          if (den > 0.f) {
            if (p.sinks) {
              const float sk = p.sinks[qh] * kLog2e;
              mul = 1.f / (den + ex2(sk - Mx));
            } else {
              mul = 1.f / den;
            }
          }
        } else {
          mul = den > 0.f ? 1.f / den : 0.f;
          if (xq == 0) p.ws_lse[(int64_t)u_split * p.R + r] = den > 0.f ? Mx + log2f(den) : -INFINITY;
        }
        const int64_t ob = ((int64_t)(b * p.Lq + qi) * p.Hq + qh) * kD + c_keep;
        // this thread's 32 columns of row r as 16-byte stores: fp32 (split record or fp32
        // output) four values per store, a 16-bit output eight
        // (a 16-bit split record takes the 16-bit path too, into the record area)
        const int64_t rec = ((int64_t)u_split * p.R + r) * kD + c_keep;
        float* dst32 = finalize ? static_cast<float*>(p.out) + ob : p.ws_o + rec;
        uint16_t* dst16 = finalize ? static_cast<uint16_t*>(p.out) + ob : reinterpret_cast<uint16_t*>(p.ws_o) + rec;
        const bool out16 = finalize ? p.out_dtype != TLLM_F32 : p.rec_type != TLLM_RECORD_F32;
        const bool bf = finalize ? p.out_dtype == TLLM_BF16 : p.rec_type == TLLM_RECORD_BF16;
        uint32_t pk[4];
#pragma unroll
        for (int i4 = 0; i4 < 8; i4++) {
          const float4 a = *chunk(xB, L, c_keep / 4 + i4);
          const float4 c = *chunk(xC, r, c_keep / 4 + i4);
          const float4 v = make_float4((__uint_as_float(o[4 * i4]) * g0 + a.x + c.x) * mul,
                                       (__uint_as_float(o[4 * i4 + 1]) * g0 + a.y + c.y) * mul,
                                       (__uint_as_float(o[4 * i4 + 2]) * g0 + a.z + c.z) * mul,
                                       (__uint_as_float(o[4 * i4 + 3]) * g0 + a.w + c.w) * mul);
          if (!out16) {
            *reinterpret_cast<float4*>(dst32 + 4 * i4) = v;
          } else {
            if (bf) {
              const __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y), h1 = __floats2bfloat162_rn(v.z, v.w);
              pk[2 * (i4 & 1)] = *reinterpret_cast<const uint32_t*>(&h0);
              pk[2 * (i4 & 1) + 1] = *reinterpret_cast<const uint32_t*>(&h1);
            } else {
              const __half2 h0 = __floats2half2_rn(v.x, v.y), h1 = __floats2half2_rn(v.z, v.w);
              pk[2 * (i4 & 1)] = *reinterpret_cast<const uint32_t*>(&h0);
              pk[2 * (i4 & 1) + 1] = *reinterpret_cast<const uint32_t*>(&h1);
            }
            if (i4 & 1)
              *reinterpret_cast<uint4*>(dst16 + 4 * (i4 - 1)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();                         // item done: every copy, MMA and TMEM access drained
  // after a timed-out wait nothing more is started (copies may still be in flight); the
  // status word says the output is not valid
  if (ld_volatile_shared(abort)) break;
  }
  if (n_list < kListCap || (n_list > 0 && ld_volatile_shared(smem_u32(sm + kOffMisc + 4)))) break;
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
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

// Dimension-major V: [pages * Hkv * D rows][bs bytes], boxes of 128 rows x 16 bytes, unswizzled.
bool encode_vdm_map(CUtensorMap* map, const void* base, int64_t rows, int bs) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)bs, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)bs};
  cuuint32_t box[2] = {16, (cuuint32_t)kD};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_cache_map(CUtensorMap* map, const void* base, int64_t rows, int bs) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD};
  cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)bs};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_fp8_supports(const tllm_decode_attn_desc& d, int rows) {
  const int bs = d.block_size;
  return d.kv_dtype == TLLM_FP8_E4M3 && d.head_dim == kD && rows >= 1 && rows <= 64 &&
         (d.v_layout == TLLM_V_TOKEN_MAJOR || (d.v_layout == TLLM_V_DIM_MAJOR && bs >= 16)) &&
         (bs == 8 || bs == 16 || bs == 32 || bs == 64 || bs == 128) &&
         (int64_t)d.num_pages * d.num_kv_heads * bs < ((int64_t)1 << 31);
}

bool tc_fp8_pointers_ok(const Params& p) {
  auto al = [](const void* x) { return ((uintptr_t)x & 15) == 0; };
  return al(p.q) && al(p.k_cache) && al(p.v_cache) && al(p.k_scales) && al(p.v_scales) && al(p.out);
}

cudaError_t launch_partial_tc_fp8(const Params& p, cudaStream_t stream) {
  CUtensorMap km, vm;
  const int64_t rows = (int64_t)p.num_pages * p.Hkv * p.bs;
  if (!encode_cache_map(&km, p.k_cache, rows, p.bs) ||
      !(p.v_dim_major ? encode_vdm_map(&vm, p.v_cache, rows / p.bs * kD, p.bs) : encode_cache_map(&vm, p.v_cache, rows, p.bs)))
    return cudaErrorInvalidValue;
  auto kern = p.v_dim_major ? partial_tc_fp8_kernel<true> : partial_tc_fp8_kernel<false>;
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(kern), (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  // persistent grid: one CTA per SM (the shared memory allows one), at most one per item
  const int n_items = p.B * p.Hkv * p.num_splits;
  const int n_sm = sm_count();
  if (n_sm <= 0) return cudaErrorInvalidValue;
  dim3 grid(n_items < n_sm ? n_items : n_sm);
  kern<<<grid, kThreads, kSmemBytes, stream>>>(p, km, vm);
  return cudaGetLastError();
}

}  // namespace tllm
