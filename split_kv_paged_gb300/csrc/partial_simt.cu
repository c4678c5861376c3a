// Pipelined CUDA-core split-KV partial kernel for few packed rows (Hq/Hkv x Lq <= 8): 16-bit,
// FP8 e4m3 or INT8 KV, head_dim 64/128/256, power-of-two block size 8..128. Decode with
// plain GQA (R = G) is this shape; with so few rows per KV head a tensor-core tile would be
// mostly padding, and the kernel is bound by the HBM stream alone.
//
// It also reads a dimension-major ("transposed") V cache, [num_pages, Hkv, D, bs]: V tiles are
// staged dimension by dimension (16-byte copies of a page row) and gathered per token.
//
// One CTA = one (request, kv head, split, block of 8 packed rows), 256 threads; with at most 8
// rows there is one row block and each KV byte of the split is read once (GQA packing: "split
// packed-Q8 verifier KV scans", hipfire PR #760, Summary). More rows (the shapes no tensor-core
// kernel takes: 16-bit caches at head_dim 256) run as several row blocks, each reading the
// split's KV (the later reads mostly from L2).
//   Load:    all threads copy tile j + kStages - 1 (K rows, V rows and, for quantised KV, the
//            per-token scales) with 16-byte cp.async into a kStages-deep shared-memory ring;
//            tokens the split does not read, or on an invalid page, are zero-filled. Page
//            ids are read two tiles ahead so their latency never sits in the loop.
//   Compute: a group of D/8 lanes owns one token at a time, each lane 8 dims; the group's
//            lanes hold the query rows (pre-scaled into log2 units) and their slice of the
//            output accumulators in registers. Every group runs its own online softmax
//            over the tokens it sees (tiny-llm PR #11: per-split online (m, l, acc)).
//   Merge:   the groups' (m, l, acc) are merged once, through shared memory, into the
//            split's normalised record (or the final output when the request has one split).
#include <type_traits>

#include "common.cuh"
#include "tc_ptx.cuh"

#ifndef SIMT_STAGES
#define SIMT_STAGES 3
#endif

namespace tllm {
namespace {

constexpr int kThreads = 256, kWarps = kThreads / 32;
constexpr int kStages = SIMT_STAGES;
constexpr int kTile = 64;        // tokens per tile
constexpr int kPgSlots = kStages + 1;   // page-id slots: tile j's ids stay readable while j + kStages's are written

__device__ __forceinline__ float ex2s(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"((uint64_t)src), "r"(ok ? 16u : 0u)
               : "memory");
}
// 8-byte variant (through L1: the .cg form copies 16 bytes only)
__device__ __forceinline__ void cp_async8_zfill(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"((uint64_t)src), "r"(ok ? 8u : 0u)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Sum of RM per-row partial dot products over the group's LPT lanes, leaving lane li with the
// full sum of one row: row li / (LPT / RM). Each halving step sends half the rows to the
// partner lane and keeps the other half (log2 RM steps), then a butterfly over the LPT / RM
// lanes that share a row: RM - 1 + log2(LPT / RM) shuffles instead of RM log2(LPT).
template <int RM, int LPT>
__device__ __forceinline__ float reduce_rows(float (&v)[RM], int li) {
#pragma unroll
  for (int c = RM, d = LPT / 2; c > 1; c >>= 1, d >>= 1) {
    const bool up = (li & d) != 0;
#pragma unroll
    for (int i = 0; i < c / 2; i++) {
      const float send = up ? v[i] : v[i + c / 2];
      const float keep = up ? v[i + c / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, d);
    }
  }
  float x = v[0];
#pragma unroll
  for (int d = LPT / RM / 2; d > 0; d >>= 1) x += __shfl_xor_sync(0xffffffffu, x, d);
  return x;
}

// Eight consecutive elements of a cache row, widened to fp32 (exactly: every e4m3, int8,
// f16 and bf16 value is representable in fp32).
template <typename KT>
struct Row8;
template <>
struct Row8<__half> {
  static constexpr int kBytes = 16;
  __device__ static void get(const uint8_t* s, float (&x)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(s);
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v[i]));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
};
template <>
struct Row8<__nv_bfloat16> {
  static constexpr int kBytes = 16;
  __device__ static void get(const uint8_t* s, float (&x)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(s);
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
      x[2 * i] = __uint_as_float(v[i] << 16);
      x[2 * i + 1] = __uint_as_float(v[i] & 0xffff0000u);
    }
  }
};
template <>
struct Row8<__nv_fp8_e4m3> {
  static constexpr int kBytes = 8;
  __device__ static void get(const uint8_t* s, float (&x)[8]) {
    const uint2 w = *reinterpret_cast<const uint2*>(s);
    const uint32_t v[2] = {w.x, w.y};
#pragma unroll
    for (int i = 0; i < 2; i++) {
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        uint32_t h2;
        const uint16_t pair = (uint16_t)(v[i] >> (16 * hh));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
        x[4 * i + 2 * hh] = f.x;
        x[4 * i + 2 * hh + 1] = f.y;
      }
    }
  }
};
template <>
struct Row8<int8_t> {
  static constexpr int kBytes = 8;
  __device__ static void get(const uint8_t* s, float (&x)[8]) {
    const uint2 w = *reinterpret_cast<const uint2*>(s);
    const uint32_t v[2] = {w.x, w.y};
#pragma unroll
    for (int i = 0; i < 8; i++) x[i] = (float)(int8_t)(v[i >> 2] >> (8 * (i & 3)));
  }
};

// Eight or sixteen consecutive elements of a cache row, widened to fp32.
// one element of the cache type, widened to fp32
template <typename KT>
__device__ __forceinline__ float elt_f32(const uint8_t* s) {
  if constexpr (std::is_same<KT, __half>::value) return __half2float(*reinterpret_cast<const __half*>(s));
  else if constexpr (std::is_same<KT, __nv_bfloat16>::value)
    return __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(s) << 16);
  else if constexpr (std::is_same<KT, int8_t>::value) return (float)*reinterpret_cast<const int8_t*>(s);
  else {
    uint32_t h2;
    const uint16_t pair = *s;                              // the code in the low byte
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
    return __half2float(*reinterpret_cast<const __half*>(&h2));
  }
}

template <typename KT, int N>
__device__ __forceinline__ void load_row(const uint8_t* s, float (&x)[N]) {
  static_assert(N % 8 == 0, "whole 8-element pieces");
#pragma unroll
  for (int c = 0; c < N / 8; c++) {
    float y[8];
    Row8<KT>::get(s + c * Row8<KT>::kBytes, y);
#pragma unroll
    for (int e = 0; e < 8; e++) x[8 * c + e] = y[e];
  }
}

template <typename KT, int D, int RM>
struct Shape {
  // dims per lane: 8 (16 would halve the lanes per token, but its query and accumulator rows
  // no longer fit two CTAs' registers per SM)
  static constexpr int kDpl = 8;
  static constexpr int kLpt = D / kDpl;                    // lanes per token (8, 16, 32)
  static constexpr int kGpw = 32 / kLpt;                   // groups per warp
  static constexpr int kGroups = kWarps * kGpw;
  static constexpr int kTpg = kTile / kGroups;             // tokens per group per tile
  static constexpr int kRowBytes = D * Row8<KT>::kBytes / 8;
  static constexpr int kRowStride = kRowBytes + 16;        // padded: groups read different rows
  static constexpr bool kScaled = sizeof(KT) == 1;
  static constexpr int kStageBytes = 2 * kTile * kRowStride + (kScaled ? 2 * kTile * 4 : 0);
  static constexpr int kChunksPerRow = kRowBytes / 16;
  static constexpr int kRingBytes = kStages * kStageBytes;
  // dimension-major V in shared memory: D rows of the tile's tokens (kTile elements), the
  // 16-byte chunks of row d placed at chunk ^ ((d / 8) % kDmChunks), so that the lanes of a
  // token group, which read dims 8 li .. 8 li + 7 of one token, reach different bank groups
  static constexpr int kElt = Row8<KT>::kBytes / 8;
  static constexpr int kDmRow = kTile * kElt;                       // bytes of one dim's row
  static constexpr int kDmChunks = kDmRow / 16;                     // 16-byte chunks per row
  static_assert(D * kDmRow <= kTile * kRowStride, "a dimension-major V tile fits the V stage");
  static_assert(D * kDmChunks == kTile * kChunksPerRow, "same copy count as the token-major tile");
  static_assert(kTpg >= 1 && kTile % kGroups == 0, "tile");
  static_assert(kRingBytes >= kMaxSplits * 8 * 4, "the fused merge's weights (splits x rows) fit in the ring");
  static_assert(kTile * kChunksPerRow % kThreads == 0, "copy split");
};

template <int RM, int D>
__host__ __device__ constexpr int merge_bytes() {
  return Shape<__half, D, RM>::kGroups * RM * (D + 2) * 4;
}

template <typename KT, int D, int RM>
__host__ __device__ constexpr int simt_smem_bytes() {
  using S = Shape<KT, D, RM>;
  const int ring = S::kRingBytes;
  const int merge = merge_bytes<RM, D>();
  return (ring > merge ? ring : merge) + kPgSlots * 32 * 4 + 64;
}

// kVdm: the V cache is dimension-major (a separate instance, so the token-major one compiles as
// without it)
template <typename KT, int D, int RM, bool kVdm>
__global__ void __launch_bounds__(kThreads, RM <= 4 ? 2 : 1) partial_simt_kernel(Params p) {
  using S = Shape<KT, D, RM>;
  if (threadIdx.x == 0) pdl_launch_dependents();
  extern __shared__ __align__(16) uint8_t smem[];
  int* pg_s = reinterpret_cast<int*>(smem + (S::kRingBytes > merge_bytes<RM, D>() ? S::kRingBytes : merge_bytes<RM, D>()));
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = blockIdx.x, b = u / p.Hkv, g = u % p.Hkv, split = blockIdx.y;
  const int r0 = blockIdx.z * RM;                          // first packed row of this CTA's block
  // the block-table entries this split reads when its request has the full length (64 of them
  // from the split's share of the row), pulled into L2 while the context length is in flight:
  // the page-id loads that follow it then hit L2
  if (p.block_table && tid < 2) {
    const int per = (p.max_blocks + p.num_splits - 1) / p.num_splits;
    const int first = min(split * per + 32 * tid, p.max_blocks - 1);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.block_table + (int64_t)b * p.max_blocks + first));
  }
  const int raw_ctx = p.context_lens[b];
  const int ctx = clamp_ctx(raw_ctx, p.max_ctx);
  if (raw_ctx != ctx && tid == 0 && split == 0 && r0 == 0) atomicOr(p.status, TLLM_FLAG_CTX_CLAMPED);
  const Span sp = request_span(ctx, p.Lq, p.window, p.num_splits, p.min_chunk, p.align);
  if (split >= sp.nsplit) return;
  const int t0 = sp.base + split * sp.chunk;
  const int t1 = min(ctx, t0 + sp.chunk);
  const int vlo = max(t0, sp.lo);                          // first token this split reads
  const int n_tiles = t1 > t0 ? (t1 - t0 + kTile - 1) / kTile : 0;
  const bool finalize = sp.nsplit == 1;
  const int u_split = u * p.max_splits + split;
  const int bs = p.bs, bs_sh = __ffs(bs) - 1;
  // pages a tile touches (a tile starts on a multiple of the tile size, a page on a multiple
  // of bs; both are powers of two)
  const int ppt = kTile >= bs ? kTile >> bs_sh : 1;

  const int grp = warp * S::kGpw + lane / S::kLpt;         // token group of this lane
  const int li = lane % S::kLpt;                           // dims li*kDpl .. li*kDpl+kDpl-1

  // query rows, pre-scaled into log2 units; rows past R stay zero and never see a key
  float q[RM][S::kDpl];
  {
    VecF32<S::kDpl> qv[RM];                                // all rows' loads in flight together
#pragma unroll
    for (int r = 0; r < RM; r++) {
      const bool real = r0 + r < p.R;
      const int qi = real ? (r0 + r) / p.G : 0, h = g * p.G + (real ? (r0 + r) % p.G : 0);
      qv[r].load(p.q, p.q_dtype, ((int64_t)(b * p.Lq + qi) * p.Hq + h) * D + li * S::kDpl, real);
    }
#pragma unroll
    for (int r = 0; r < RM; r++) {
      qv[r].get(p.q_dtype, q[r]);
#pragma unroll
      for (int e = 0; e < S::kDpl; e++) q[r][e] *= p.scale_log2;
    }
  }
  // after the reduction each lane owns the softmax state of one row: rho
  constexpr int kLpr = S::kLpt / RM;                       // lanes per row
  const int rho = li / kLpr;
  const int pos_rho = r0 + rho < p.R ? ctx - p.Lq + (r0 + rho) / p.G : -1;   // its position (-1: no keys)
  const int gbase = lane - li;                             // first lane of the group

  const uint8_t* kc = static_cast<const uint8_t*>(p.k_cache);
  const uint8_t* vc = static_cast<const uint8_t*>(p.v_cache);
  // page id of slot i of tile jt (-1: not read / invalid), read by threads i < ppt
  auto page_of = [&](int jt, int i) -> int {
    const int first = t0 + jt * kTile + i * bs;         // first token of the slot
    if (jt >= n_tiles || first >= t1 || first + bs <= vlo) return -1;
    const int pg = page_at(p, b, first >> bs_sh);
    if (pg < 0 || pg >= p.num_pages) {
      atomicOr(p.status, TLLM_FLAG_BAD_PAGE);
      return -1;
    }
    return pg;
  };
  // issue the copies of tile jt into stage jt % kStages (page ids already in pg_s)
  auto issue = [&](int jt) {
    const int st = jt % kStages;
    const uint32_t kdst = sbase + st * S::kStageBytes, vdst = kdst + kTile * S::kRowStride;
    const int tt = t0 + jt * kTile;
    // consecutive threads copy consecutive 16-byte chunks (coalesced rows)
#pragma unroll
    for (int i = 0; i < kTile * S::kChunksPerRow / kThreads; i++) {
      const int c = tid + i * kThreads;
      const int tok = c / S::kChunksPerRow, off = (c % S::kChunksPerRow) * 16;
      const int t = tt + tok;
      const int pg = pg_s[(jt % kPgSlots) * 32 + (tok >> bs_sh)];
      const bool ok = jt < n_tiles && pg >= 0 && t >= vlo && t < t1;
      const int64_t row = ok ? ((int64_t)pg * p.Hkv + g) * bs + (t & (bs - 1)) : 0;
      cp_async16_zfill(kdst + tok * S::kRowStride + off, kc + row * S::kRowBytes + off, ok);
      if constexpr (!kVdm) {
        cp_async16_zfill(vdst + tok * S::kRowStride + off, vc + row * S::kRowBytes + off, ok);
      } else {
        // dimension-major V: chunk c is 16 bytes of dim d's page row, tokens tl .. tl + 16 / kElt
        // - 1 of the tile (on one page when bs is a multiple of 16 / kElt; else, 8-token pages of
        // an 8-bit cache, its two 8-byte halves come from two pages); a piece any of whose tokens
        // the split reads is copied whole, the rest zero-filled
        constexpr int kTpc = 16 / S::kElt;
        const int d = c / S::kDmChunks, cc = c % S::kDmChunks, tl = cc * kTpc;
        const uint32_t vd = vdst + d * S::kDmRow + ((cc ^ ((d >> 3) & (S::kDmChunks - 1))) << 4);
        const int np = bs < kTpc ? 2 : 1, tpp = kTpc / np;     // pieces of the chunk, tokens each
        for (int h = 0; h < np; h++) {
          const int tlh = tl + h * tpp, tv = tt + tlh;
          const int pgv = pg_s[(jt % kPgSlots) * 32 + (tlh >> bs_sh)];
          const bool okv = jt < n_tiles && pgv >= 0 && tv + tpp > vlo && tv < t1;
          const int64_t src = okv ? ((((int64_t)pgv * p.Hkv + g) * D + d) * bs + (tv & (bs - 1))) * S::kElt : 0;
          if (np == 1) cp_async16_zfill(vd, vc + src, okv);
          else cp_async8_zfill(vd + 8 * h, vc + src, okv);
        }
      }
    }
    if constexpr (S::kScaled) {
      const uint32_t sdst = vdst + kTile * S::kRowStride;   // [K scales | V scales], kTile each
      for (int c = tid; c < 2 * (kTile / 4); c += kThreads) {
        const int which = c / (kTile / 4), tok = (c % (kTile / 4)) * 4;
        const int t = tt + tok;
        const int pg = pg_s[(jt % kPgSlots) * 32 + (tok >> bs_sh)];
        // four tokens share a page (bs >= 8); a partly read quad is copied whole and the
        // unread tokens are masked by position when scores are formed
        const bool ok = jt < n_tiles && pg >= 0 && t + 3 >= vlo && t < t1;
        const int64_t row = ok ? ((int64_t)pg * p.Hkv + g) * bs + (t & (bs - 1)) : 0;
        cp_async16_zfill(sdst + which * kTile * 4 + tok * 4, (which ? p.v_scales : p.k_scales) + row, ok);
      }
    }
  };

  // prologue: page ids of tiles 0 .. kStages - 1 published, tile kStages's in a register
  for (int jt = 0; jt < kStages; jt++)
    if (tid < ppt) pg_s[(jt % kPgSlots) * 32 + tid] = page_of(jt, tid);
  int pg_next = tid < ppt ? page_of(kStages, tid) : -1;
  __syncthreads();
  for (int jt = 0; jt < kStages - 1; jt++) {
    issue(jt);
    cp_async_commit();
  }

  float m_row = -INFINITY, l_row = 0.f, acc[RM][S::kDpl];
#pragma unroll
  for (int r = 0; r < RM; r++)
#pragma unroll
    for (int e = 0; e < S::kDpl; e++) acc[r][e] = 0.f;
  const int pos_lo = ctx - p.Lq;                           // lowest real row position

  for (int j = 0; j < n_tiles; j++) {
    cp_async_wait<kStages - 2>();
    // tile j landed; stage (j - 1) % kStages is free; the page ids of tile j + kStages - 1,
    // written during tile j - 1, are visible
    __syncthreads();
    {
      const int jn = j + kStages - 1;                      // refill the stage freed by tile j - 1
      if (jn < n_tiles) issue(jn);
      cp_async_commit();                                   // (empty past the end: keeps the count)
      // ids of tile j + kStages for the next iteration (slot not read before then)
      if (tid < ppt) pg_s[((j + kStages) % kPgSlots) * 32 + tid] = pg_next;
      pg_next = tid < ppt ? page_of(j + kStages + 1, tid) : -1;
    }
    const int st = j % kStages;
    const uint8_t* ks_tile = smem + st * S::kStageBytes;
    const uint8_t* vs_tile = ks_tile + kTile * S::kRowStride;
    const float* sc = reinterpret_cast<const float*>(vs_tile + kTile * S::kRowStride);
    const int tt = t0 + j * kTile;
    // a tile every row sees whole (every token read, on a valid page, at or before every
    // row's position and inside every row's window) needs no per-token mask
    bool pages_ok = true;
    const int* pgt = pg_s + (j % kPgSlots) * 32;         // page ids of tile j
    for (int i = 0; i < ppt; i++) pages_ok = pages_ok && pgt[i] >= 0;
    const bool whole = pages_ok && tt >= vlo && tt + kTile <= t1 && tt + kTile - 1 <= pos_lo &&
                       (p.window <= 0 || tt > ctx - 1 - p.window);
    if constexpr (kVdm) {
      // V of the tokens the split does not read (before the window, past the length, on a page
      // not loaded) may hold stale or poisoned values in a partly read chunk: zero them before
      // the PV reads the tile (their p is 0, but 0 x NaN is not 0)
      if (!(pages_ok && tt >= vlo && tt + kTile <= t1)) {
        uint8_t* vw = smem + st * S::kStageBytes + kTile * S::kRowStride;
        for (int idx = tid; idx < D * kTile; idx += kThreads) {
          const int d = idx / kTile, tl = idx % kTile, t = tt + tl;
          if (!(t >= vlo && t < t1 && pgt[kTile >= bs ? tl >> bs_sh : 0] >= 0)) {
            uint8_t* e = vw + d * S::kDmRow + ((((tl * S::kElt) >> 4) ^ ((d >> 3) & (S::kDmChunks - 1))) << 4) +
                         ((tl * S::kElt) & 15);
            if constexpr (S::kElt == 2) *reinterpret_cast<uint16_t*>(e) = 0;
            else *e = 0;
          }
        }
        __syncthreads();
      }
    }
    float sk[S::kTpg];                                        // this lane's row: scores of the group's tokens
#pragma unroll
    for (int k = 0; k < S::kTpg; k++) {
      const int tok = grp * S::kTpg + k, t = tt + tok;
      float kx[S::kDpl];
      load_row<KT, S::kDpl>(ks_tile + tok * S::kRowStride + li * (S::kRowBytes / S::kLpt), kx);
      float dot[RM];
#pragma unroll
      for (int r = 0; r < RM; r++) {
        float2 a = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < S::kDpl; e += 2)
          a = ptx::ffma2(make_float2(q[r][e], q[r][e + 1]), make_float2(kx[e], kx[e + 1]), a);
        dot[r] = a.x + a.y;
      }
      const float x = reduce_rows<RM, S::kLpt>(dot, li);
      const float ksc = S::kScaled ? sc[tok] : 1.f;
      const bool vis = whole || (t >= vlo && t < t1 && pgt[tok >> bs_sh] >= 0 && t <= pos_rho &&
                                 (p.window <= 0 || pos_rho - t < p.window));
      sk[k] = vis ? x * ksc : -INFINITY;
    }
    // online softmax of this group over its kTpg tokens, for this lane's row
    float mx = sk[0];
#pragma unroll
    for (int k = 1; k < S::kTpg; k++) mx = fmaxf(mx, sk[k]);
    const float m_new = fmaxf(m_row, mx);
    const float alpha = m_new == m_row ? 1.f : (m_row == -INFINITY ? 0.f : ex2s(m_row - m_new));
    m_row = m_new;
    float pk[S::kTpg];
    l_row *= alpha;
#pragma unroll
    for (int k = 0; k < S::kTpg; k++) {
      pk[k] = m_new == -INFINITY ? 0.f : ex2s(sk[k] - m_new);
      l_row += pk[k];
    }
    // every lane holds accumulators of every row: rescale factors and weights are broadcast
    // from the lanes that own the rows
    if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
      for (int r = 0; r < RM; r++) {
        const float a_r = __shfl_sync(0xffffffffu, alpha, gbase + r * kLpr);
#pragma unroll
        for (int e = 0; e < S::kDpl; e++) acc[r][e] *= a_r;
      }
    }
#pragma unroll
    for (int k = 0; k < S::kTpg; k++) {
      const int tok = grp * S::kTpg + k;
      float vx[S::kDpl];
      if constexpr (!kVdm) {
        load_row<KT, S::kDpl>(vs_tile + tok * S::kRowStride + li * (S::kRowBytes / S::kLpt), vx);
      } else {
        // dims 8 li .. 8 li + 7 of token tok: one element from each of 8 dim rows (their chunk
        // placed at chunk ^ li)
        const uint8_t* vr = vs_tile + ((((tok * S::kElt) >> 4) ^ (li & (S::kDmChunks - 1))) << 4) +
                            ((tok * S::kElt) & 15);
#pragma unroll
        for (int e = 0; e < S::kDpl; e++) vx[e] = elt_f32<KT>(vr + (S::kDpl * li + e) * S::kDmRow);
      }
      // masked tokens have p = 0; their scale may be anything (NaN included), so it is
      // selected away rather than multiplied
      const float vsc = S::kScaled ? sc[kTile + tok] : 1.f;
#pragma unroll
      for (int r = 0; r < RM; r++) {
        const float p_r = __shfl_sync(0xffffffffu, pk[k], gbase + r * kLpr);
        const float w = p_r != 0.f ? p_r * vsc : 0.f;
#pragma unroll
        for (int e = 0; e < S::kDpl; e += 2) {
          const float2 y = ptx::ffma2(make_float2(w, w), make_float2(vx[e], vx[e + 1]),
                                      make_float2(acc[r][e], acc[r][e + 1]));
          acc[r][e] = y.x;
          acc[r][e + 1] = y.y;
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();                                         // ring free: reuse it for the merge

  // merge: group states -> [grp][r][D] accumulators and [grp][r] (m, l)
  float* mo = reinterpret_cast<float*>(smem);                        // [kGroups][RM][D]
  float* ml = mo + S::kGroups * RM * D;                              // [kGroups][RM][2]
#pragma unroll
  for (int r = 0; r < RM; r++) {
#pragma unroll
    for (int e = 0; e < S::kDpl; e += 4)
      *reinterpret_cast<float4*>(mo + ((grp * RM + r) * D + li * S::kDpl + e)) =
          make_float4(acc[r][e], acc[r][e + 1], acc[r][e + 2], acc[r][e + 3]);
  }
  if (li % kLpr == 0) {
    ml[(grp * RM + rho) * 2] = m_row;
    ml[(grp * RM + rho) * 2 + 1] = l_row;
  }
  __syncthreads();
  for (int idx = tid; idx < RM * D; idx += kThreads) {
    const int r = idx / D, d = idx % D, rg = r0 + r;     // row in the block, packed row
    if (rg >= p.R) continue;
    float M = -INFINITY;
    for (int gi = 0; gi < S::kGroups; gi++) M = fmaxf(M, ml[(gi * RM + r) * 2]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int gi = 0; gi < S::kGroups; gi++) {
        const float mg = ml[(gi * RM + r) * 2];
        const float w = mg == -INFINITY ? 0.f : ex2s(mg - M);
        L = fmaf(w, ml[(gi * RM + r) * 2 + 1], L);
        O = fmaf(w, mo[(gi * RM + r) * D + d], O);
      }
    }
    const int qi = rg / p.G, h = g * p.G + rg % p.G;
    if (finalize) {
      float den = L;
      if (p.sinks && M != -INFINITY) den += ex2s(p.sinks[h] * kLog2e - M);
      store_f32(p.out, p.out_dtype, ((int64_t)(b * p.Lq + qi) * p.Hq + h) * D + d, L > 0.f ? O / den : 0.f);
    } else {
      store_rec(p, ((int64_t)u_split * p.R + rg) * D + d, L > 0.f ? O / L : 0.f);
      if (d == 0) p.ws_lse[(int64_t)u_split * p.R + rg] = L > 0.f ? M + log2f(L) : -INFINITY;
    }
  }
  // fused combine: the CTA that completes the request's records merges them into the output
  // (planned only with one row block)
  if (!finalize && p.fused && gridDim.z == 1) {
    __shared__ int last_arrival;
    __syncthreads();                                       // the merge area below is free again
    fused_combine_arrive(p, u, b, g, sp.nsplit, &last_arrival, reinterpret_cast<float*>(smem));
  }
}

template <typename KT, int D, int RM, bool kVdm>
cudaError_t launch_one(const Params& p, dim3 grid, cudaStream_t stream) {
  constexpr int smem = simt_smem_bytes<KT, D, RM>();
  const void* f = reinterpret_cast<const void*>(&partial_simt_kernel<KT, D, RM, kVdm>);
  cudaError_t e = set_smem_attr(f, smem);
  if (e != cudaSuccess) return e;
  partial_simt_kernel<KT, D, RM, kVdm><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <typename KT, int RM, bool kVdm>
cudaError_t launch_d(const Params& p, dim3 grid, cudaStream_t stream) {
  switch (p.D) {
    case 64: return launch_one<KT, 64, RM, kVdm>(p, grid, stream);
    case 128: return launch_one<KT, 128, RM, kVdm>(p, grid, stream);
    case 256: return launch_one<KT, 256, RM, kVdm>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int RM, bool kVdm>
cudaError_t launch_kt(const Params& p, dim3 grid, cudaStream_t stream) {
  switch (p.kv_dtype) {
    case TLLM_F16: return launch_d<__half, RM, kVdm>(p, grid, stream);
    case TLLM_BF16: return launch_d<__nv_bfloat16, RM, kVdm>(p, grid, stream);
    case TLLM_FP8_E4M3: return launch_d<__nv_fp8_e4m3, RM, kVdm>(p, grid, stream);
    case TLLM_INT8: return launch_d<int8_t, RM, kVdm>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool simt_supports(const tllm_decode_attn_desc& d, int rows) {
  const int bs = d.block_size;
  const bool kv_ok = d.kv_dtype == TLLM_F16 || d.kv_dtype == TLLM_BF16 || d.kv_dtype == TLLM_FP8_E4M3 ||
                     d.kv_dtype == TLLM_INT8;
  const bool v_ok = d.v_layout == TLLM_V_TOKEN_MAJOR || d.v_layout == TLLM_V_DIM_MAJOR;
  return kv_ok && v_ok && (d.head_dim == 64 || d.head_dim == 128 || d.head_dim == 256) &&
         rows >= 1 && (bs == 8 || bs == 16 || bs == 32 || bs == 64 || bs == 128);
}

int simt_tile(int) { return kTile; }

bool simt_pointers_ok(const Params& p) {
  auto al = [](const void* x) { return ((uintptr_t)x & 15) == 0; };
  return al(p.q) && al(p.k_cache) && al(p.v_cache) && (p.k_scales == nullptr || (al(p.k_scales) && al(p.v_scales)));
}

cudaError_t launch_partial_simt(const Params& p, cudaStream_t stream) {
  // rows per CTA (a transposed V cache: always 8, one instance per cache type and head_dim)
  const int rm = p.R <= 4 && !p.v_dim_major ? 4 : 8;
  dim3 grid(p.B * p.Hkv, p.num_splits, (p.R + rm - 1) / rm);
  if (p.v_dim_major) return launch_kt<8, true>(p, grid, stream);
  return rm == 4 ? launch_kt<4, false>(p, grid, stream) : launch_kt<8, false>(p, grid, stream);
}

}  // namespace tllm
