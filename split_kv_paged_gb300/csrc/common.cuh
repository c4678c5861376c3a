// Shared definitions of the GB300 split-KV decode attention kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tllm_decode_attn.h"

#define TLLM_HD __host__ __device__ __forceinline__

namespace tllm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSplits = 256;     // aiter PR #5628, Changes: partition limit of 256

// Everything a partial or combine launch needs; built by the host from the plan and
// the call arguments.
struct Params {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;       // [B, max_blocks] or nullptr (contiguous cache)
  const int32_t* context_lens;
  const float* k_scales;            // [num_pages, Hkv, bs] or nullptr
  const float* v_scales;
  const float* sinks;               // [Hq] or nullptr
  void* out;
  uint32_t* status;                 // workspace status word
  uint32_t* counters;               // [B*Hkv] arrival counters of the fused combine
  float* ws_lse;                    // [B*Hkv][max_splits][R]
  float* ws_o;                      // [B*Hkv][max_splits][R][D] in rec_type (fp32, or 16-bit viewed through it)
  int B, Lq, Hq, Hkv, G, D, R, bs;
  int max_blocks, num_pages, window, num_splits, max_splits, min_chunk, align;
  int max_ctx;                      // max_blocks * bs: lengths are clamped to it
  float scale_log2;                 // softmax scale * log2(e)
  int q_dtype, kv_dtype, out_dtype;
  int v_dim_major;                  // v_cache [num_pages, Hkv, D, bs] (TLLM_V_DIM_MAJOR)
  int rec_type;                     // tllm_record_type of the split records
  int fused;                        // the partial kernel merges the splits (no combine launch)
  int test_stall;                   // failure-detection tests: the widening kernel issues no QK^T
};

// Element i of the split-record area: fp32, or bf16 / f16 when the plan asked for 16-bit records.
__device__ __forceinline__ void store_rec(const Params& p, int64_t i, float v) {
  if (p.rec_type == TLLM_RECORD_F32) p.ws_o[i] = v;
  else if (p.rec_type == TLLM_RECORD_BF16) reinterpret_cast<__nv_bfloat16*>(p.ws_o)[i] = __float2bfloat16_rn(v);
  else reinterpret_cast<__half*>(p.ws_o)[i] = __float2half_rn(v);
}
// Four consecutive record elements from i (i a multiple of 4): one 16- or 8-byte store.
__device__ __forceinline__ void store_rec4(const Params& p, int64_t i, float4 v) {
  if (p.rec_type == TLLM_RECORD_F32) {
    *reinterpret_cast<float4*>(p.ws_o + i) = v;
  } else if (p.rec_type == TLLM_RECORD_BF16) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.ws_o) + i) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  } else {
    const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(p.ws_o) + i) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  }
}

// ---- the split rule (host and device) -------------------------------------------
// tiny-llm PR #11, design section: each partial CTA derives its own logical range
// from the device-side visible length, chunk = ceil(visible / splits). Here the
// visible range of a request is the union of its rows' ranges, [lo, ctx), with
// lo = ctx - Lq + 1 - W under a window W (aiter PR #5628, Changes: windowed work is
// capped by the causal-window union and tile alignment). Split boundaries are
// measured from base = lo rounded down to `align` (a page / tile multiple), so every
// split starts on an aligned token.

struct Span {
  int lo;      // first key any row of the request may see
  int base;    // lo rounded down to align
  int ctx;     // clamped context length (one past the last key)
  int chunk;   // tokens per split
  int nsplit;  // splits this request uses (>= 1)
};

TLLM_HD int clamp_ctx(int ctx, int max_ctx) { return ctx < 0 ? 0 : (ctx > max_ctx ? max_ctx : ctx); }

TLLM_HD Span request_span(int ctx, int Lq, int window, int num_splits, int min_chunk, int align) {
  Span s;
  s.ctx = ctx;
  int lo = 0;
  if (window > 0) {
    lo = ctx - Lq + 1 - window;
    if (lo < 0) lo = 0;
  }
  if (lo > ctx) lo = ctx;
  s.lo = lo;
  s.base = (lo / align) * align;
  int vis = ctx - s.base;
  int c = num_splits > 0 ? (vis + num_splits - 1) / num_splits : vis;
  if (c < min_chunk) c = min_chunk;
  c = ((c + align - 1) / align) * align;
  if (c < align) c = align;
  s.chunk = c;
  int n = (vis + c - 1) / c;
  s.nsplit = n < 1 ? 1 : n;
  return s;
}

// ---- page lookup ----------------------------------------------------------------------
// Physical page of block `blk` of request b: the block table's entry, or, for a contiguous
// cache (no block table: "split-KV decode attention design record", tiny-llm PR #11, design
// section, the ContiguousRows address mode), block blk of request b is page
// b * max_blocks + blk, so the cache is [batch][max_blocks][Hkv][bs][D] in one piece.
__device__ __forceinline__ int page_at(const Params& p, int b, int blk) {
  return p.block_table ? __ldg(p.block_table + (int64_t)b * p.max_blocks + blk) : b * p.max_blocks + blk;
}

// ---- the work list of the persistent partial kernels ----------------------------------
// The real items of a call are the (unit = request x kv head, split) pairs with split below
// the number of splits the unit's request uses (from its device-side length), in unit-major
// order; CTA c of a grid of G CTAs takes the items of rank c, c + G, c + 2 G, ... So every CTA
// gets real work while there is any, and a request's unused split slots cost nothing (aiter
// PR #5628, Changes: a work plan built on the GPU from the lengths, with capacity fixed for
// graph replay).
//
// build_work_list writes into shared memory the items of this CTA whose rank lies in
// [round0, round0 + kListCap) of its own sequence: entry i is (unit << 8) | split of the
// item of rank c + G (round0 + i), and entry kListCap + i the request's context length as
// read from context_lens (not yet clamped). It returns how many items it wrote (the same value
// in every thread). Every thread of the CTA calls it; it ends with a CTA barrier, after which
// the list is read-only until the next call. `list` holds kListWords ints: the two arrays and
// one int of scan scratch per warp.
constexpr int kListCap = 64;
constexpr int kListWords = 2 * kListCap + 32;

__device__ __forceinline__ int build_work_list(const Params& p, int* list, int round0) {
  int* scan = list + 2 * kListCap;
  const int nthr = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
  const int G = gridDim.x, c = blockIdx.x;
  const int U = p.B * p.Hkv;
  int base = 0;                                     // real items in the units before this chunk
  for (int u0 = 0; u0 < U; u0 += nthr) {
    const int u = u0 + tid;
    int n = 0, raw = 0;
    if (u < U) {
      raw = p.context_lens[u / p.Hkv];
      n = request_span(clamp_ctx(raw, p.max_ctx), p.Lq, p.window, p.num_splits, p.min_chunk, p.align).nsplit;
    }
    int incl = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) scan[warp] = incl;
    __syncthreads();
    int wofs = 0, total = 0;
    for (int w = 0; w < nwarps; w++) {
      const int v = scan[w];
      wofs += w < warp ? v : 0;
      total += v;
    }
    const int first = base + wofs + incl - n;       // rank of (u, split 0)
    int k = first + ((c - first % G) % G + G) % G;  // smallest rank >= first owned by this CTA
    for (; k < first + n; k += G) {
      const int i = k / G - round0;
      if (i >= 0 && i < kListCap) {
        list[i] = (u << 8) | (k - first);
        list[kListCap + i] = raw;
      }
    }
    base += total;
    __syncthreads();                                // scan reused; the list complete after the last chunk
  }
  const int mine = base > c ? (base - c + G - 1) / G : 0;
  const int left = mine - round0;
  return left < 0 ? 0 : (left > kListCap ? kListCap : left);
}

// ---- element conversions ---------------------------------------------------------

template <typename T> struct DT;
template <> struct DT<__half> { static constexpr int code = TLLM_F16; };
template <> struct DT<__nv_bfloat16> { static constexpr int code = TLLM_BF16; };
template <> struct DT<float> { static constexpr int code = TLLM_F32; };

struct e4m3_t { uint8_t x; };
struct i8_t { int8_t x; };

__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(e4m3_t v) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(v.x, __NV_E4M3);
  return __half2float(__half(h));
}
__device__ __forceinline__ float to_f32(i8_t v) { return (float)v.x; }

// Runtime-typed load / store for the few elements touched once per CTA (queries,
// outputs): keeps the template count down to the hot-loop types.
__device__ __forceinline__ float load_f32(const void* base, int dtype, int64_t i) {
  switch (dtype) {
    case TLLM_F16: return __half2float(static_cast<const __half*>(base)[i]);
    case TLLM_BF16: return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
    default: return static_cast<const float*>(base)[i];
  }
}
// N consecutive elements (N a multiple of 8) of a runtime-typed array (f16, bf16 or f32),
// fetched as 16-byte pieces that are all in flight before any is used, then widened to fp32.
// Element i must start on a 16-byte boundary.
template <int N>
struct VecF32 {
  static_assert(N % 8 == 0, "whole 16-byte pieces");
  uint4 raw[N / 4];                                  // f32 needs N / 4 pieces, 16-bit types N / 8
  __device__ __forceinline__ void load(const void* base, int dtype, int64_t i, bool valid) {
    const bool f32 = dtype == TLLM_F32;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(base) + i * (f32 ? 4 : 2));
#pragma unroll
    for (int c = 0; c < N / 4; c++)
      raw[c] = (valid && (f32 || c < N / 8)) ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
  }
  __device__ __forceinline__ void get(int dtype, float (&x)[N]) const {
    if (dtype == TLLM_F32) {
#pragma unroll
      for (int c = 0; c < N / 4; c++) {
        x[4 * c] = __uint_as_float(raw[c].x);
        x[4 * c + 1] = __uint_as_float(raw[c].y);
        x[4 * c + 2] = __uint_as_float(raw[c].z);
        x[4 * c + 3] = __uint_as_float(raw[c].w);
      }
    } else {
      const bool bf = dtype == TLLM_BF16;
#pragma unroll
      for (int c = 0; c < N / 8; c++) {
        const uint32_t w[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
          float2 f;
          if (bf) {
            f = make_float2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u));
          } else {
            f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
          }
          x[8 * c + 2 * k] = f.x;
          x[8 * c + 2 * k + 1] = f.y;
        }
      }
    }
  }
};

__device__ __forceinline__ void store_f32(void* base, int dtype, int64_t i, float v) {
  switch (dtype) {
    case TLLM_F16: static_cast<__half*>(base)[i] = __float2half_rn(v); break;
    case TLLM_BF16: static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v); break;
    default: static_cast<float*>(base)[i] = v; break;
  }
}

__device__ __forceinline__ void store_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__half* p, float v) { *p = __float2half_rn(v); }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// ---- the fused combine -----------------------------------------------------------------
// Record element i, read through L2 (written by other CTAs of the same launch).
__device__ __forceinline__ float load_rec(const Params& p, int64_t i) {
  if (p.rec_type == TLLM_RECORD_F32) return __ldcg(p.ws_o + i);
  const unsigned short h = __ldcg(reinterpret_cast<const unsigned short*>(p.ws_o) + i);
  return p.rec_type == TLLM_RECORD_BF16 ? __uint_as_float((uint32_t)h << 16)
                                        : __half2float(__ushort_as_half(h));
}

// One CTA merges the n split records of unit u (request b, kv head g) into the output: per
// packed row the max-LSE-stabilised weighted sum over the splits in split order, with the sink
// once in the denominator, rows that saw no key zero; the same arithmetic as the combine kernel
// ("split-KV decode attention design record", tiny-llm PR #11, open question 1: the last CTA
// of a request merges its partials; "split packed-Q8 verifier KV scans", hipfire PR #760,
// Summary: stable max-LSE merge). Every thread of the CTA calls it. `wsm` is shared scratch of
// at least n * R floats: the LSEs are read once into it and turned into normalised weights per
// row, then every output element loads all its records at once (their latencies overlap).
__device__ __forceinline__ void merge_unit(const Params& p, int u, int b, int g, int n, float* wsm) {
  const int D = p.D, R = p.R;
  const float* lse = p.ws_lse + (int64_t)u * p.max_splits * R;
  for (int i = threadIdx.x; i < n * R; i += blockDim.x) wsm[i] = __ldcg(lse + i);   // [s][r]
  __syncthreads();
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    float M = -INFINITY;
    for (int s = 0; s < n; s++) M = fmaxf(M, wsm[s * R + r]);
    float den = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < n; s++) den += exp2f(wsm[s * R + r] - M);   // 0 for a split with no key
      if (p.sinks) {
        const float sk = p.sinks[g * p.G + r % p.G] * kLog2e, M2 = fmaxf(M, sk);
        den = den * exp2f(M - M2) + exp2f(sk - M2);
        M = M2;
      }
    }
    for (int s = 0; s < n; s++) wsm[s * R + r] = M == -INFINITY ? 0.f : exp2f(wsm[s * R + r] - M) / den;
  }
  __syncthreads();
  const int64_t rec0 = (int64_t)u * p.max_splits * R * D;
  for (int idx = threadIdx.x; idx < R * D; idx += blockDim.x) {
    const int r = idx / D, d = idx % D;
    float acc = 0.f;
    for (int s0 = 0; s0 < n; s0 += 8) {
      float x[8];
#pragma unroll
      for (int k = 0; k < 8; k++)
        x[k] = s0 + k < n && wsm[(s0 + k) * R + r] != 0.f ? load_rec(p, rec0 + ((int64_t)(s0 + k) * R + r) * D + d) : 0.f;
#pragma unroll
      for (int k = 0; k < 8; k++)
        if (s0 + k < n) acc = fmaf(wsm[(s0 + k) * R + r], x[k], acc);
    }
    store_f32(p.out, p.out_dtype, ((int64_t)(b * p.Lq + r / p.G) * p.Hq + g * p.G + r % p.G) * D + d, acc);
  }
}

// Called by every thread of a CTA that has just written the split record of unit u (stores
// issued, not yet fenced): the CTA whose record completes the request's n records (an arrival
// ticket on the unit's counter, which wraps back to zero on that last arrival, so nothing
// waits and the counter is ready for the next call) merges them. `flag` is a shared int, `wsm`
// shared scratch of n * R floats.
__device__ __forceinline__ void fused_combine_arrive(const Params& p, int u, int b, int g, int n, int* flag,
                                                     float* wsm) {
  __threadfence();                                   // this CTA's records, visible GPU-wide
  __syncthreads();
  if (threadIdx.x == 0) *flag = atomicInc(p.counters + u, (unsigned)(n - 1)) == (unsigned)(n - 1);
  __syncthreads();
  if (*flag) {
    __threadfence();                                 // every other record, seen after the ticket
    merge_unit(p, u, b, g, n, wsm);
  }
}

// Programmatic dependent launch: a partial kernel lets the combine grid be scheduled as soon
// as all its CTAs have started (the combine's CTAs then sit on free SM slots, so its launch
// latency overlaps the partial's tail); the combine waits for the partial grid to complete,
// with its memory visible, before it reads the records.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Raise a kernel's dynamic shared-memory limit once per device (the attribute is
// per function and device; calling it again is harmless but costs a driver call).
cudaError_t set_smem_attr(const void* func, int bytes);
// Streaming multiprocessors of the current device (cached per device); 0 on error.
int sm_count();

// Checks the arguments of a call (tllm_decode_attn_splitkv and its stages) against the plan in
// `ws` and fills the launch parameters; queues nothing and makes no CUDA call.
tllm_status make_params(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                        const int32_t* context_lens, int32_t query_len, const float* kv_scales,
                        const float* sinks, int32_t window, int32_t num_splits, const tllm_workspace* ws,
                        void* out, Params* p);

// ---- launchers (one per kernel family) ---------------------------------------------
cudaError_t launch_partial_generic(const Params& p, cudaStream_t stream);
cudaError_t launch_combine(const Params& p, cudaStream_t stream);
bool generic_supports(const tllm_decode_attn_desc& d, int rows);
cudaError_t launch_partial_tc_fp8(const Params& p, cudaStream_t stream);
bool simt_supports(const tllm_decode_attn_desc& d, int rows);
int simt_tile(int head_dim);
bool simt_pointers_ok(const Params& p);
cudaError_t launch_partial_simt(const Params& p, cudaStream_t stream);
bool tc_i8_supports(const tllm_decode_attn_desc& d, int rows);
bool tc_i8_pointers_ok(const Params& p);
cudaError_t launch_partial_tc_i8(const Params& p, cudaStream_t stream);
bool tc_fp8_supports(const tllm_decode_attn_desc& d, int rows);
bool tc_fp8_pointers_ok(const Params& p);
bool tc_b16_supports(const tllm_decode_attn_desc& d, int rows);
bool tc_b16_pointers_ok(const Params& p);
cudaError_t launch_partial_tc_b16(const Params& p, cudaStream_t stream);

}  // namespace tllm
