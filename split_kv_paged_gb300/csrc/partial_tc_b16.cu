// 16-bit tensor-core split-KV partial kernel for sm_103a (tcgen05 kind::f16): f16 or bf16 KV
// read as loaded, a query of the same type, head_dim 128, up to 16 packed rows per KV head
// (the decode shapes: GQA groups x a few query rows), block size 8..128.
//
// With so few rows per KV head, a row-major tile would leave the MMA's M dimension nearly
// empty and put the softmax on a handful of threads. So both contractions run transposed,
// with the tokens on M:
//   S^T = K Q^T:     A = the K tile as loaded (128 tokens x 128 dims, K-major, 128-byte
//                    swizzle, 64-dim halves), B = Q (16 rows, zero-padded, K-major);
//                    D = S^T in TMEM, lane = token, column = row.
//   O^T += V^T P^T:  A = the V tile as loaded, read MN-major (M = dims), B = P^T (K-major,
//                    32 rows: P_hi then P_lo, columns = tokens); D = O^T in TMEM, lane = dim.
// P is sent as a 16-bit high part plus the 16-bit rounding of its remainder, so the product
// carries about 16 significant bits of P (a bare bf16 P would round it to 8).
//
// Persistent CTAs, one per SM, take the real (request x kv head, split) items of a work list
// built on the device from the lengths, in turn (item k to CTA k mod grid); per item each
// KV page of the split is read from HBM once (GQA packing: "split packed-Q8 verifier KV
// scans", hipfire PR #760, Summary). Roles (256 threads):
//   warp 0      K producer, warp 2 V producer: page ids one group of tiles ahead, one TMA box
//               per (page, 64-dim half) into 3-stage rings of 128-token tiles;
//   warp 1      one thread issues every S^T MMA; warp 3 one thread issues every O^T MMA;
//   warps 4..7  softmax, thread = token of the tile (TMEM lane). A row's maximum is reduced
//               per warp (redux.sync) and across the 4 warps through shared memory; P goes to
//               shared memory as the B operand of the tile's O^T MMA. Online softmax in log2
//               units (tiny-llm PR #11: per-split online (m, l, acc)); a row's exponent
//               reference moves only when a tile's maximum passes it by more than kSlack, so
//               O^T is rarely rescaled. Each thread keeps the row sums of its own token lane;
//               they are reduced once, in the epilogue, where the same threads read O^T
//               (thread = dim) and store every row as whole lines.
//
// Every wait is bounded in time; a timeout sets TLLM_FLAG_TIMEOUT, lets every role run to its
// end without waiting, drains the copies and MMAs in flight, skips the output stores, takes
// no further item and frees TMEM.
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace tllm {
namespace {

using namespace ptx;

constexpr int kTile = 128;                           // tokens per tile (M of S^T)
constexpr int kD = 128;                              // head_dim (M of O^T)
constexpr int kStages = 3;
constexpr int kThreads = 256;
constexpr int kNq = 16;                              // N of S^T: packed rows, zero-padded
constexpr int kNp = 32;                              // N of O^T: P_hi rows 0..15, P_lo rows 16..31
constexpr float kSlack = 2.f;
constexpr uint32_t kFull = 0xffffffffu;

// shared memory (byte offsets from a 1024-aligned base)
constexpr uint32_t kHalf = kTile * 128;              // one 64-dim half of a tile: 128 tokens x 128 B
constexpr uint32_t kStageBytes = 2 * kHalf;          // 32 KB
constexpr uint32_t kOffV = kStages * kStageBytes;
constexpr uint32_t kOffQ = 2 * kOffV;                // Q: [2 dim halves][16 rows][128 B]
constexpr uint32_t kQHalf = kNq * 128;
constexpr uint32_t kOffP = kOffQ + 2 * kQHalf;       // P^T: 2 buffers x [2 token halves][32 rows][128 B]
constexpr uint32_t kPHalf = kNp * 128;
constexpr uint32_t kPBuf = 2 * kPHalf;
constexpr uint32_t kOffX = kOffP + 2 * kPBuf;        // exchange: [2][4 warps][16] maxima, [4][16] sums
constexpr uint32_t kOffBar = kOffX + 1024;
constexpr uint32_t kNumBars = 4 * kStages + 4 * 2 + 2;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kOffList = kOffMisc + 64;            // work list + its scan scratch
constexpr uint32_t kSmemBytes = kOffList + kListWords * 4 + 1024;   // + alignment slack
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kPHalf % 1024 == 0, "operand alignment");
static_assert(kSmemBytes <= 232448, "shared memory");

// TMEM columns: S^T buffer s at 16 s, O^T at 32 (P_hi rows, then P_lo rows)
constexpr uint32_t kTmemCols = 64, kColS = 0, kColO = 32;

__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t byte) {
  return (row >> 3) * 1024 + (row & 7) * 128 + ((((byte >> 4) ^ row) & 7) << 4) + (byte & 15);
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// maximum over the 32 lanes of the (fully active) warp
__device__ __forceinline__ float warp_max(float x) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}
// a float -> the 16-bit KV type (bits), round to nearest; and back
template <bool BF> __device__ __forceinline__ uint16_t to16(float x) {
  if constexpr (BF) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  else return __half_as_ushort(__float2half_rn(x));
}
template <bool BF> __device__ __forceinline__ float from16(uint16_t h) {
  if constexpr (BF) return __uint_as_float((uint32_t)h << 16);
  else return __half2float(__ushort_as_half(h));
}
__device__ __forceinline__ void st_shared_u16(uint32_t a, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"(v) : "memory");
}

constexpr uint32_t kBarKFull = 0, kBarKEmpty = kStages, kBarVFull = 2 * kStages, kBarVEmpty = 3 * kStages,
                   kBarSFull = 4 * kStages, kBarSFree = kBarSFull + 2, kBarPFull = kBarSFree + 2,
                   kBarPvDone = kBarPFull + 2, kBarQFull = kBarPvDone + 2, kBarMmaFin = kBarQFull + 1;
static_assert(kBarMmaFin + 1 == kNumBars, "barrier count");
struct Bars {
  uint32_t base;
  __device__ uint32_t at(uint32_t i) const { return base + 8u * i; }
  __device__ uint32_t k_full(int s) const { return at(kBarKFull + s); }     // K producer -> S^T MMA (tx bytes)
  __device__ uint32_t k_empty(int s) const { return at(kBarKEmpty + s); }   // S^T MMA done with the K stage
  __device__ uint32_t v_full(int s) const { return at(kBarVFull + s); }     // V producer -> O^T MMA (tx bytes)
  __device__ uint32_t v_empty(int s) const { return at(kBarVEmpty + s); }   // O^T MMA done with the V stage
  __device__ uint32_t s_full(int b) const { return at(kBarSFull + b); }     // S^T buffer b written
  __device__ uint32_t s_free(int b) const { return at(kBarSFree + b); }     // S^T buffer b read out
  __device__ uint32_t p_full(int b) const { return at(kBarPFull + b); }     // P^T buffer b written, O^T rescaled
  __device__ uint32_t pv_done(int b) const { return at(kBarPvDone + b); }   // O^T MMA of a tile of parity b done
  __device__ uint32_t q_full() const { return at(kBarQFull); }              // Q in shared memory
  __device__ uint32_t mma_fin() const { return at(kBarMmaFin); }            // final commits of the two issuers
};

__device__ __forceinline__ void set_abort(uint32_t abort, uint32_t* status) {
  if (!ld_volatile_shared(abort)) {
    asm volatile("st.volatile.shared.b32 [%0], %1;" ::"r"(abort), "r"(1) : "memory");
    atomicOr(status, TLLM_FLAG_TIMEOUT);
  }
}

// NR: packed rows rounded up to 4, 8 or 16; BF: bf16 (else f16) query and cache
template <int NR, bool BF>
__global__ void __launch_bounds__(kThreads)
    partial_tc_b16_kernel(const Params p, const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) pdl_launch_dependents();
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffMisc);
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  // P^T rows that no thread writes (NR..15 of each part) stay zero for the whole launch
  for (uint32_t i = tid; i < 2 * kPBuf / 16; i += kThreads)
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(sbase + kOffP + 16 * i), "r"(0));
  fence_proxy_async();
  // The first work list is built while the TMEM allocation completes: its barriers also
  // publish the TMEM address.
  int* wlist = reinterpret_cast<int*>(sm + kOffList);
  tc_fence_before();
  const int n_list0 = build_work_list(p, wlist, 0);
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Bars bars{sbase + kOffBar};
  const uint32_t abort = sbase + kOffMisc + 4;

  // the real (request x kv head, split) items of the work list, in turn
  int n_list = n_list0;
  for (int round0 = 0;; round0 += kListCap) {
  if (round0 > 0) n_list = build_work_list(p, wlist, round0);
  for (int li = 0; li < n_list; li++) {
  const int u = wlist[li] >> 8, b = u / p.Hkv, g = u % p.Hkv, split = wlist[li] & 255;
  const int raw_ctx = wlist[kListCap + li];
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
  const int bs_sh = __ffs(bs) - 1;                   // bs is a power of two, 8..128
  const int ppt_sh = 7 - bs_sh, ppt = 1 << ppt_sh;   // pages per tile (1..16)
  const int gt_sh = 5 - ppt_sh, gt = 1 << gt_sh;     // tiles per group of 32 page ids
  // page ids of a group of tiles, one per lane (lane = tile of the group x page slot)
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
  int pg_cur = 0, nd_cur = 0, pg_nxt = 0, nd_nxt = 0;
  if (warp == 0 || warp == 2) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(warp == 0 ? &kmap : &vmap)) : "memory");
    fetch(0, pg_cur, nd_cur);
    fetch(1, pg_nxt, nd_nxt);
  }

  if (tid == 0) {
    for (int s = 0; s < kStages; s++) {
      mbar_init(bars.k_full(s), 1);
      mbar_init(bars.k_empty(s), 1);
      mbar_init(bars.v_full(s), 1);
      mbar_init(bars.v_empty(s), 1);
    }
    for (int s = 0; s < 2; s++) {
      mbar_init(bars.s_full(s), 1);
      mbar_init(bars.s_free(s), 4);        // one elected lane per softmax warp
      mbar_init(bars.p_full(s), 4);
      mbar_init(bars.pv_done(s), 1);
    }
    mbar_init(bars.q_full(), 4);
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
    // lane = (64-dim half, page slot): lanes [0, ppt) copy half 0 of the tile's pages,
    // [ppt, 2 ppt) half 1
    const bool isk = warp == 0;
    const uint32_t full = isk ? bars.k_full(0) : bars.v_full(0);
    const uint32_t empty = isk ? bars.k_empty(0) : bars.v_empty(0);
    const uint32_t ring = sbase + (isk ? 0u : kOffV);
    const CUtensorMap* map = isk ? &kmap : &vmap;
    const int slot = lane & (ppt - 1), half = lane >> ppt_sh;
    int issued = 0;
    for (int j = 0; j < n_tiles; j++) {
      if (j > 0 && (j & (gt - 1)) == 0) {
        pg_cur = pg_nxt;
        nd_cur = nd_nxt;
        fetch((j >> gt_sh) + 1, pg_nxt, nd_nxt);
      }
      const int st = j % kStages;
      if (j >= kStages && !mbar_wait(empty + 8 * st, ((j / kStages) - 1) & 1, abort)) set_abort(abort, p.status);
      if (ld_volatile_shared(abort)) break;
      const int src = (((j & (gt - 1)) << ppt_sh) + slot) & 31;
      const int pgv = __shfl_sync(kFull, pg_cur, src);
      const int ndv = __shfl_sync(kFull, nd_cur, src);
      int page = -1;
      if (half < 2 && ndv) {
        if (pgv < 0 || pgv >= p.num_pages) {
          if (isk && half == 0) atomicOr(p.status, TLLM_FLAG_BAD_PAGE);
        } else {
          page = pgv;
        }
      }
      const uint32_t m = __ballot_sync(kFull, page >= 0);
      if (lane == 0) mbar_arrive_expect_tx(full + 8 * st, __popc(m) * (uint32_t)bs * 128u);
      __syncwarp();
      if (page >= 0) {
        const int64_t row = ((int64_t)page * p.Hkv + g) * bs;
        tma_load_2d(ring + st * kStageBytes + half * kHalf + slot * bs * 128, map, half * 64, (int)row,
                    full + 8 * st);
      }
      issued = j + 1;
    }
    // drain: every issued stage's copies must land before the item ends
    for (int j = max(0, issued - kStages); j < issued; j++)
      if (!mbar_wait(full + 8 * (j % kStages), (j / kStages) & 1, 0u)) set_abort(abort, p.status);
    // ... and the release of each of those stages by its MMA (an asynchronous tcgen05.commit
    // arrival) must have landed too, before the next item re-initialises the barriers
    for (int j = max(0, issued - kStages); j < issued; j++)
      if (!mbar_wait(empty + 8 * (j % kStages), (j / kStages) & 1, abort)) set_abort(abort, p.status);
   } else if (lane == 0) {
    // ---------------- MMA issuers: warp 1 every S^T, warp 3 every O^T ----------------
    bool ok = true;
    if (warp == 1) {
      const uint32_t idqk = idesc_f16(128, kNq, BF ? 1 : 0, 0, 0);
      ok = mbar_wait(bars.q_full(), 0, abort);
      for (int j = 0; ok && j < n_tiles; j++) {
        const int st = j % kStages, sb = j & 1;
        if (!mbar_wait(bars.k_full(st), (j / kStages) & 1, abort)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(bars.s_free(sb), ((j >> 1) - 1) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kt = sbase + st * kStageBytes;
#pragma unroll
        for (int k = 0; k < kD / 16; k++)
          mma_f16_ss(tmem + kColS + 16 * sb, sdesc_sw128(kt + (k >> 2) * kHalf + 32 * (k & 3), 16, 1024),
                     sdesc_sw128(sbase + kOffQ + (k >> 2) * kQHalf + 32 * (k & 3), 16, 1024), idqk, k > 0 ? 1u : 0u);
        mma_commit(bars.s_full(sb));
        mma_commit(bars.k_empty(st));
      }
    } else {
      const uint32_t idpv = idesc_f16(128, kNp, BF ? 1 : 0, 1, 0);
      for (int j = 0; ok && j < n_tiles; j++) {
        const int pb = j & 1, st = j % kStages;
        if (!mbar_wait(bars.p_full(pb), (j >> 1) & 1, abort)) { ok = false; break; }
        if (!mbar_wait(bars.v_full(st), (j / kStages) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t vt = sbase + kOffV + st * kStageBytes;
        const uint32_t pt = sbase + kOffP + pb * kPBuf;
#pragma unroll
        for (int k = 0; k < kTile / 16; k++)
          mma_f16_ss(tmem + kColO, sdesc_sw128(vt + 2048 * k, kHalf, 1024),
                     sdesc_sw128(pt + (k >> 2) * kPHalf + 32 * (k & 3), 16, 1024), idpv, (j > 0 || k > 0) ? 1u : 0u);
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
    // ---------------- softmax: thread = token L of the tile (TMEM lane); in the epilogue, dim L ----------------
    const int wq = warp & 3;
    const int L = 32 * wq + lane;
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    float* xm = reinterpret_cast<float*>(sm + kOffX);          // [2][4][16] partial row maxima
    float* xl = xm + 2 * 4 * 16;                               // [4][16] partial row sums

    // Q rows -> shared memory in the B-operand layout; rows R..15 zero
#pragma unroll
    for (int c2 = 0; c2 < 2; c2++) {
      const int c = L + 128 * c2, n = c >> 4, d0 = (c & 15) * 8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (n < p.R) {
        const int qi = n / p.G, qh = g * p.G + n % p.G;
        v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                 ((int64_t)(b * p.Lq + qi) * p.Hq + qh) * kD + d0));
      }
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sbase + kOffQ + (d0 >> 6) * kQHalf +
                                                                      sw128(n, (d0 & 63) * 2)),
                   "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
    }
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.q_full());

    int pos[NR];                                             // position of each packed row (-1: padding)
#pragma unroll
    for (int r = 0; r < NR; r++) pos[r] = r < p.R ? ctx - p.Lq + r / p.G : -1;
    float M[NR], l[NR];
#pragma unroll
    for (int r = 0; r < NR; r++) {
      M[r] = -INFINITY;
      l[r] = 0.f;
    }
    // this thread's token of tile jt: its page id, or -1 when the split does not read it
    auto tok_page = [&](int jt) -> int {
      const int t = t0 + jt * kTile + L;
      return (jt < n_tiles && t >= sp.lo && t < t1) ? page_at(p, b, t >> bs_sh) : -1;
    };
    int pg_tok = tok_page(0);
    const int last = n_tiles - 1;
    for (int j = 0; j < n_tiles; j++) {
      const int st = j % kStages, sb = j & 1;
      const int t = t0 + j * kTile + L;
      const bool rd = pg_tok >= 0 && pg_tok < p.num_pages;    // token read (and its page in the pool)
      pg_tok = tok_page(j + 1);
      if (!mbar_wait(bars.s_full(sb), (j >> 1) & 1, abort)) set_abort(abort, p.status);
      tc_fence_after();
      uint32_t s[16];
      tmem_ld16(tmem + lane_off + kColS + 16 * sb, s);
      if (!rd) {
        // a token this split does not read: its V row becomes zero, so stale or poisoned bytes
        // never reach the O^T MMA (published to it by the p_full arrival, after a proxy fence)
        if (!mbar_wait(bars.v_full(st), (j / kStages) & 1, abort)) set_abort(abort, p.status);
        const uint32_t vrow = sbase + kOffV + st * kStageBytes;
#pragma unroll
        for (int hf = 0; hf < 2; hf++)
#pragma unroll
          for (int c = 0; c < 8; c++)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(vrow + hf * kHalf + sw128(L, 16 * c)), "r"(0));
      }
      tmem_ld_wait16(s);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.s_free(sb));

      // scores in log2 units, masked: causal among the rows, window, tokens not read
      float x[NR];
#pragma unroll
      for (int r = 0; r < NR; r++) {
        const bool vis = rd && t <= pos[r] && (p.window <= 0 || pos[r] - t < p.window);
        x[r] = vis ? __uint_as_float(s[r]) * p.scale_log2 : -INFINITY;
      }
      float* xs = xm + (j & 1) * 64;
#pragma unroll
      for (int r = 0; r < NR; r++) {
        const float mw = warp_max(x[r]);
        if (lane == 0) xs[16 * wq + r] = mw;
      }
      named_bar(1, 128);
      bool moved = false;
      float alpha[NR], pr[NR];
#pragma unroll
      for (int r = 0; r < NR; r++) {
        const float mx = fmaxf(fmaxf(xs[r], xs[16 + r]), fmaxf(xs[32 + r], xs[48 + r]));
        const float Mn = mx > M[r] + kSlack ? mx : M[r];
        alpha[r] = Mn == -INFINITY ? 1.f : ex2(M[r] - Mn);
        moved |= alpha[r] != 1.f;
        M[r] = Mn;
        pr[r] = Mn == -INFINITY ? 0.f : ex2(x[r] - Mn);
        l[r] = l[r] * alpha[r] + pr[r];
      }
      // this P^T buffer is free once the O^T MMA of tile j - 2 is done
      if (j >= 2 && !mbar_wait(bars.pv_done(sb), ((j - 2) >> 1) & 1, abort)) set_abort(abort, p.status);
      const uint32_t pcol = sbase + kOffP + sb * kPBuf + (L >> 6) * kPHalf;
      const uint32_t pbyte = (L & 63) * 2;
#pragma unroll
      for (int r = 0; r < NR; r++) {
        const uint16_t hi = to16<BF>(pr[r]);
        const uint16_t lo = to16<BF>(pr[r] - from16<BF>(hi));
        st_shared_u16(pcol + sw128(r, pbyte), hi);
        st_shared_u16(pcol + sw128(kNq + r, pbyte), lo);
      }
      fence_proxy_async();
      // a row reference moved: O^T (this thread: dim L, every row) holds tiles < j, so it is
      // rescaled once the O^T MMA of tile j - 1 is done (the same for every thread)
      if (moved && j >= 1) {
        if (!mbar_wait(bars.pv_done((j - 1) & 1), ((j - 1) >> 1) & 1, abort)) set_abort(abort, p.status);
        tc_fence_after();
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + kColO, o);
        tmem_ld_wait();
#pragma unroll
        for (int r = 0; r < NR; r++) {
          o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
          o[kNq + r] = __float_as_uint(__uint_as_float(o[kNq + r]) * alpha[r]);
        }
        tmem_st32(tmem + lane_off + kColO, o);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.p_full(sb));
    }

    // ---------------- epilogue: row sums, O^T (thread = dim L), normalised rows ----------------
    if (!mbar_wait(bars.pv_done(last & 1), (last >> 1) & 1, abort)) set_abort(abort, p.status);
    tc_fence_after();
#pragma unroll
    for (int r = 0; r < NR; r++) {
      float v = l[r];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
      if (lane == 0) xl[16 * wq + r] = v;
    }
    named_bar(1, 128);
    uint32_t o[32];
    tmem_ld32(tmem + lane_off + kColO, o);
    tmem_ld_wait();
    if (!ld_volatile_shared(abort)) {
#pragma unroll
      for (int r = 0; r < NR; r++) {
        if (r < p.R) {
          const float den = (xl[r] + xl[16 + r]) + (xl[32 + r] + xl[48 + r]);
          const float val = __uint_as_float(o[r]) + __uint_as_float(o[kNq + r]);
          const int qi = r / p.G, qh = g * p.G + r % p.G;
          if (finalize) {
            float mul = 0.f;
            if (den > 0.f) mul = 1.f / (p.sinks ? den + ex2(p.sinks[qh] * kLog2e - M[r]) : den);
            store_f32(p.out, p.out_dtype, ((int64_t)(b * p.Lq + qi) * p.Hq + qh) * kD + L, val * mul);
          } else {
            store_rec(p, ((int64_t)u_split * p.R + r) * kD + L, den > 0.f ? val / den : 0.f);
            if (L == 0) p.ws_lse[(int64_t)u_split * p.R + r] = den > 0.f ? M[r] + log2f(den) : -INFINITY;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();                         // item done: every copy, MMA and TMEM access drained
  if (ld_volatile_shared(abort)) break;
  }
  if (n_list < kListCap || (n_list > 0 && ld_volatile_shared(abort))) break;
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder_b16() {
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

// [rows][128] 16-bit elements, one box = 64 elements (128 B) x bs rows, 128-byte swizzle
bool encode_b16_map(CUtensorMap* map, const void* base, int64_t rows, int bs) {
  auto enc = get_encoder_b16();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)bs};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NR, bool BF>
cudaError_t launch_nr(const Params& p, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t stream) {
  auto kern = partial_tc_b16_kernel<NR, BF>;
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(kern), (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_items = p.B * p.Hkv * p.num_splits;
  const int n_sm = sm_count();
  if (n_sm <= 0) return cudaErrorInvalidValue;
  dim3 grid(n_items < n_sm ? n_items : n_sm);
  kern<<<grid, kThreads, kSmemBytes, stream>>>(p, km, vm);
  return cudaGetLastError();
}

template <bool BF>
cudaError_t launch_bf(const Params& p, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t stream) {
  if (p.R <= 4) return launch_nr<4, BF>(p, km, vm, stream);
  if (p.R <= 8) return launch_nr<8, BF>(p, km, vm, stream);
  return launch_nr<16, BF>(p, km, vm, stream);
}

}  // namespace

bool tc_b16_supports(const tllm_decode_attn_desc& d, int rows) {
  const int bs = d.block_size;
  return (d.kv_dtype == TLLM_F16 || d.kv_dtype == TLLM_BF16) && d.q_dtype == d.kv_dtype && d.head_dim == kD &&
         d.v_layout == TLLM_V_TOKEN_MAJOR &&
         rows >= 1 && rows <= kNq && (bs == 8 || bs == 16 || bs == 32 || bs == 64 || bs == 128) &&
         (int64_t)d.num_pages * d.num_kv_heads * bs < ((int64_t)1 << 31);
}

bool tc_b16_pointers_ok(const Params& p) {
  auto al = [](const void* x) { return ((uintptr_t)x & 15) == 0; };
  return al(p.q) && al(p.k_cache) && al(p.v_cache);
}

cudaError_t launch_partial_tc_b16(const Params& p, cudaStream_t stream) {
  CUtensorMap km, vm;
  const int64_t rows = (int64_t)p.num_pages * p.Hkv * p.bs;
  if (!encode_b16_map(&km, p.k_cache, rows, p.bs) || !encode_b16_map(&vm, p.v_cache, rows, p.bs))
    return cudaErrorInvalidValue;
  if (p.R < 1 || p.R > kNq || p.D != kD) return cudaErrorInvalidValue;
  return p.kv_dtype == TLLM_BF16 ? launch_bf<true>(p, km, vm, stream) : launch_bf<false>(p, km, vm, stream);
}

}  // namespace tllm
