// Combine kernel: merges the split records of each request with a max-LSE-stabilised
// weighted sum ("split-KV decode attention design record", tiny-llm PR #11: the
// flash-decoding merge; "split packed-Q8 verifier KV scans", hipfire PR #760:
// stable max-LSE reduction), visiting only the splits the request actually used
// ("tune MTP work budgets and planned reduction", aiter PR #5628, Changes), and
// applying the sink logit once, in the denominator.
//
// A CTA of 8 warps takes 8 / WPR packed rows of one (request, kv head); WPR warps share a row
// and take its splits in turn (warp w of the row: splits w, w + WPR, ...), so a request with
// many splits is merged by many warps at once. A lane holds D / 32 consecutive columns, so a
// split's record row is one coalesced load of the warp. A warp loads the records of up to kG
// of its splits before using any (their latencies overlap) and merges groups online: the running
// maximum only grows, earlier groups are rescaled by 2^(M_old - M_new). Each split's weight is
// computed once, by the lane holding its LSE, and broadcast. The WPR partial results of a row
// (maximum, denominator, weighted sum) are merged through shared memory in warp order, so the
// result does not depend on timing. Records are fp32, LSE in log2 units. The kernel is
// launched as a programmatic dependent of the partial kernel and waits on it before reading
// the records, so its launch overlaps the partial's tail.
#include <type_traits>

#include "common.cuh"

namespace tllm {
namespace {

constexpr int kWarps = 8;

// V consecutive elements of a record row (fp32, bf16 or f16), widened to fp32
template <int V, typename RT>
struct VecF {
  float v[V];
  __device__ __forceinline__ void load(const RT* x) {
    if constexpr (sizeof(RT) == 4) {
#pragma unroll
      for (int c = 0; c < V; c += (V < 4 ? V : 4)) {
        if constexpr (V >= 4) {
          const float4 a = *reinterpret_cast<const float4*>(x + c);
          v[c] = a.x; v[c + 1] = a.y; v[c + 2] = a.z; v[c + 3] = a.w;
        } else {
          const float2 a = *reinterpret_cast<const float2*>(x);
          v[0] = a.x; v[1] = a.y;
        }
      }
    } else {
      // V 16-bit values: 4 bytes (V = 2), 8 (V = 4) or 16 (V = 8) in one load
      uint32_t w[V / 2];
      if constexpr (V == 8) {
        const uint4 a = *reinterpret_cast<const uint4*>(x);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
      } else if constexpr (V == 4) {
        const uint2 a = *reinterpret_cast<const uint2*>(x);
        w[0] = a.x; w[1] = a.y;
      } else {
        w[0] = *reinterpret_cast<const uint32_t*>(x);
      }
#pragma unroll
      for (int c = 0; c < V / 2; c++) {
        float2 f;
        if constexpr (std::is_same<RT, __nv_bfloat16>::value)
          f = make_float2(__uint_as_float(w[c] << 16), __uint_as_float(w[c] & 0xffff0000u));
        else
          f = __half22float2(*reinterpret_cast<const __half2*>(&w[c]));
        v[2 * c] = f.x;
        v[2 * c + 1] = f.y;
      }
    }
  }
};

// V output elements from fp32 values: one 8- or 16-byte store for 16-bit outputs
template <typename OT, int V>
__device__ __forceinline__ void store_row(OT* out, const float* a, float mul) {
  if constexpr (sizeof(OT) == 4) {
    if constexpr (V >= 4) {
#pragma unroll
      for (int c = 0; c < V; c += 4)
        *reinterpret_cast<float4*>(out + c) = make_float4(a[c] * mul, a[c + 1] * mul, a[c + 2] * mul, a[c + 3] * mul);
    } else {
#pragma unroll
      for (int c = 0; c < V; c++) store_out(out + c, a[c] * mul);
    }
  } else {
    uint32_t w[V / 2];
#pragma unroll
    for (int c = 0; c < V; c += 2) {
      if constexpr (std::is_same<OT, __nv_bfloat16>::value) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a[c] * mul, a[c + 1] * mul);
        w[c / 2] = *reinterpret_cast<const uint32_t*>(&h);
      } else {
        const __half2 h = __floats2half2_rn(a[c] * mul, a[c + 1] * mul);
        w[c / 2] = *reinterpret_cast<const uint32_t*>(&h);
      }
    }
    if constexpr (V == 8) {
      *reinterpret_cast<uint4*>(out) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if constexpr (V == 4) {
      *reinterpret_cast<uint2*>(out) = make_uint2(w[0], w[1]);
    } else {
      *reinterpret_cast<uint32_t*>(out) = w[0];
    }
  }
}

// D columns, WPR warps per row, kG splits per load group, RT the record element type
template <typename OT, int D, int WPR, int kG, typename RT>
__global__ void __launch_bounds__(kWarps * 32) combine_kernel(Params p) {
  constexpr int V = D / 32;                      // columns per lane
  constexpr int RPC = kWarps / WPR;              // rows per CTA
  static_assert(kG <= 32, "one LSE per lane");
  __shared__ float xm[kWarps], xd[kWarps];
  __shared__ __align__(16) float xa[WPR > 1 ? kWarps * D : 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rsub = warp / WPR, wsub = warp % WPR;
  const int r = blockIdx.y * RPC + rsub;
  const int u = blockIdx.x, b = u / p.Hkv, g = u % p.Hkv;
  const int ctx = clamp_ctx(p.context_lens[b], p.max_ctx);
  const Span sp = request_span(ctx, p.Lq, p.window, p.num_splits, p.min_chunk, p.align);
  if (sp.nsplit <= 1) return;                    // (the whole CTA: one request) finalised by the partial
  const int n = sp.nsplit;
  const bool live = r < p.R;
  const int col = V * lane;
  pdl_wait();                                    // the partial grid's records are complete
  const int rr = live ? r : 0;
  const float* lse = p.ws_lse + (int64_t)u * p.max_splits * p.R + rr;
  const RT* o = reinterpret_cast<const RT*>(p.ws_o) + ((int64_t)u * p.max_splits * p.R + rr) * D + col;
  const int64_t stride = (int64_t)p.R * D;

  // this warp's splits: wsub, wsub + WPR, ...; lane k of a group holds the LSE of its k-th split
  float M = -INFINITY, den = 0.f, a[V];
#pragma unroll
  for (int c = 0; c < V; c++) a[c] = 0.f;
  const int mine = live && wsub < n ? (n - wsub + WPR - 1) / WPR : 0;
  for (int k0 = 0; k0 < mine; k0 += kG) {
    const int sl = wsub + (k0 + lane) * WPR;
    const float ls = lane < kG && k0 + lane < mine ? lse[(int64_t)sl * p.R] : -INFINITY;
    VecF<V, RT> x[kG];
#pragma unroll
    for (int k = 0; k < kG; k++)
      if (k0 + k < mine) x[k].load(o + (int64_t)(wsub + (k0 + k) * WPR) * stride);
    float mg = fmaxf(M, ls);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, off));
    if (mg == -INFINITY) continue;               // no split so far saw a key
    const float sc = exp2f(M - mg);              // 0 while M = -inf (den and a are 0 then)
    M = mg;
    const float wl = exp2f(ls - M);
    float dl = wl;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, off);
    den = den * sc + dl;
#pragma unroll
    for (int c = 0; c < V; c++) a[c] *= sc;
    // a split with weight 0 (LSE -inf) contributes exactly nothing, whatever its record holds
#pragma unroll
    for (int k = 0; k < kG; k++) {
      const float w = __shfl_sync(0xffffffffu, wl, k);
      if (k0 + k < mine) {
#pragma unroll
        for (int c = 0; c < V; c++) a[c] = w != 0.f ? fmaf(w, x[k].v[c], a[c]) : a[c];
      }
    }
  }
  if constexpr (WPR > 1) {
    // merge the row's WPR partials in warp order
    if (lane == 0) {
      xm[warp] = M;
      xd[warp] = den;
    }
#pragma unroll
    for (int c = 0; c < V; c++) xa[warp * D + col + c] = a[c];
    __syncthreads();
    if (wsub != 0) return;
    float Mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < WPR; w++) Mx = fmaxf(Mx, xm[warp + w]);
    M = Mx;
    den = 0.f;
#pragma unroll
    for (int c = 0; c < V; c++) a[c] = 0.f;
    if (Mx != -INFINITY) {
#pragma unroll
      for (int w = 0; w < WPR; w++) {
        const float f = exp2f(xm[warp + w] - Mx);   // 0 for a warp that saw no key
        den = fmaf(f, xd[warp + w], den);
        const float* xs = xa + (warp + w) * D + col;
#pragma unroll
        for (int c = 0; c < V; c++) a[c] = f != 0.f ? fmaf(f, xs[c], a[c]) : a[c];
      }
    }
  }
  if (!live) return;
  const int i = r / p.G, h = g * p.G + r % p.G;
  OT* out = static_cast<OT*>(p.out) + ((int64_t)(b * p.Lq + i) * p.Hq + h) * D + col;
  if (M == -INFINITY) {                          // no split saw a key: zero row
#pragma unroll
    for (int c = 0; c < V; c++) a[c] = 0.f;
    store_row<OT, V>(out, a, 0.f);
    return;
  }
  if (p.sinks) {
    const float sk = p.sinks[h] * kLog2e;
    const float M2 = fmaxf(M, sk);
    const float sc = exp2f(M - M2);
    den = den * sc + exp2f(sk - M2);
#pragma unroll
    for (int c = 0; c < V; c++) a[c] *= sc;
  }
  store_row<OT, V>(out, a, 1.f / den);
}

// launched with programmatic stream serialisation: it may start while the partial kernel
// before it in the stream finishes, and waits on that grid inside (pdl_wait)
template <typename K>
cudaError_t launch_pdl(K kernel, dim3 grid, cudaStream_t stream, const Params& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Warps per row from the plan's split count: one warp per row while a request has at most 8
// splits (its records are one load group), more as the splits grow, so that each warp loads
// about one group.
template <typename OT, int D, int WPR>
cudaError_t launch_wpr(const Params& p, cudaStream_t stream) {
  constexpr int kG = D >= 256 ? 4 : 8;
  const dim3 grid(p.B * p.Hkv, (p.R + kWarps / WPR - 1) / (kWarps / WPR));
  switch (p.rec_type) {
    case TLLM_RECORD_BF16: return launch_pdl(combine_kernel<OT, D, WPR, kG, __nv_bfloat16>, grid, stream, p);
    case TLLM_RECORD_F16: return launch_pdl(combine_kernel<OT, D, WPR, kG, __half>, grid, stream, p);
    default: return launch_pdl(combine_kernel<OT, D, WPR, kG, float>, grid, stream, p);
  }
}

template <typename OT, int D>
cudaError_t launch_combine_d(const Params& p, cudaStream_t stream) {
  const int s = p.num_splits;
  if (s <= 8) return launch_wpr<OT, D, 1>(p, stream);
  if (s <= 16) return launch_wpr<OT, D, 2>(p, stream);
  if (s <= 32) return launch_wpr<OT, D, 4>(p, stream);
  return launch_wpr<OT, D, 8>(p, stream);
}

template <typename OT>
cudaError_t launch_combine_t(const Params& p, cudaStream_t stream) {
  switch (p.D) {
    case 64: return launch_combine_d<OT, 64>(p, stream);
    case 128: return launch_combine_d<OT, 128>(p, stream);
    case 256: return launch_combine_d<OT, 256>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_combine(const Params& p, cudaStream_t stream) {
  switch (p.out_dtype) {
    case TLLM_F32: return launch_combine_t<float>(p, stream);
    case TLLM_BF16: return launch_combine_t<__nv_bfloat16>(p, stream);
    case TLLM_F16: return launch_combine_t<__half>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tllm
