// Generic split-KV partial kernel on CUDA cores: any supported dtype combination,
// head_dim 64/128/256, any block size. It is the correctness baseline every faster
// variant is compared with, and the fallback for shapes they do not cover.
//
// It also reads a dimension-major ("transposed") V cache, [num_pages, Hkv, D, bs].
//
// One CTA = one (request, kv head, split, block of 16 packed rows). The packed rows of
// a KV head are its G query heads times the Lq query rows (GQA packing: "split packed-Q8
// verifier KV scans", hipfire PR #760, Summary). The CTA walks its split's tokens in
// tiles of 32 through the block table, runs an online softmax per row in log2 units and
// emits either the final output (the request has one split) or a normalised record.
#include "common.cuh"

namespace tllm {
namespace {

constexpr int kThreads = 128;
constexpr int kRows = 16;    // packed rows per CTA
constexpr int kTile = 32;    // tokens per tile (one per lane in the score phase)

template <typename KT, int D>
__global__ void __launch_bounds__(kThreads) partial_generic_kernel(Params p) {
  if (threadIdx.x == 0) pdl_launch_dependents();
  extern __shared__ float smem[];
  float* q_s = smem;                                   // [kRows][D]
  float* k_s = q_s + kRows * D;                        // [kTile][D + 1]
  float* v_s = k_s + kTile * (D + 1);                  // [kTile][D]
  float* p_s = v_s + kTile * D;                        // [kRows][kTile]
  float* ks_s = p_s + kRows * kTile;                   // [kTile]
  float* vs_s = ks_s + kTile;                          // [kTile]
  float* alpha_s = vs_s + kTile;                       // [kRows]
  float* m_s = alpha_s + kRows;                        // [kRows]
  float* l_s = m_s + kRows;                            // [kRows]
  int64_t* row_s = reinterpret_cast<int64_t*>(l_s + kRows + (kRows & 1 ? 1 : 0));  // [kTile]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = blockIdx.x, b = u / p.Hkv, g = u % p.Hkv, split = blockIdx.y;
  const int r0 = blockIdx.z * kRows;

  const int raw_ctx = p.context_lens[b];
  const int ctx = clamp_ctx(raw_ctx, p.max_ctx);
  if (raw_ctx != ctx && tid == 0 && split == 0 && blockIdx.z == 0) atomicOr(p.status, TLLM_FLAG_CTX_CLAMPED);
  const Span sp = request_span(ctx, p.Lq, p.window, p.num_splits, p.min_chunk, p.align);
  if (split >= sp.nsplit) return;
  const int t0 = sp.base + split * sp.chunk;
  const int t1 = min(ctx, t0 + sp.chunk);
  const bool finalize = sp.nsplit == 1;

  // Query rows, pre-scaled into log2 units.
  for (int idx = tid; idx < kRows * D; idx += kThreads) {
    int j = idx / D, d = idx % D, r = r0 + j;
    float v = 0.f;
    if (r < p.R) {
      int i = r / p.G, h = g * p.G + r % p.G;
      v = load_f32(p.q, p.q_dtype, ((int64_t)(b * p.Lq + i) * p.Hq + h) * D + d) * p.scale_log2;
    }
    q_s[idx] = v;
  }
  // Per-row softmax state, owned by warp (row % 4), replicated across its lanes.
  float m_run[kRows / 4], l_run[kRows / 4];
  int pos[kRows / 4];
  for (int k = 0; k < kRows / 4; k++) {
    m_run[k] = -INFINITY;
    l_run[k] = 0.f;
    int r = r0 + warp + 4 * k;
    pos[k] = r < p.R ? ctx - p.Lq + r / p.G : -1;   // row position; -1 never sees a key
  }
  constexpr int DC = (D + kThreads - 1) / kThreads;   // output columns per thread
  float acc[kRows][DC];
  for (int j = 0; j < kRows; j++)
    for (int c = 0; c < DC; c++) acc[j][c] = 0.f;

  const KT* kc = static_cast<const KT*>(p.k_cache);
  const KT* vc = static_cast<const KT*>(p.v_cache);
  for (int tt = t0; tt < t1; tt += kTile) {
    __syncthreads();
    if (tid < kTile) {                                 // page walk for the tile
      int t = tt + tid;
      int64_t row = -1;
      float ks = 0.f, vs = 0.f;
      if (t >= sp.lo && t < t1) {                      // keys below the window are never read
        int page = page_at(p, b, t / p.bs);
        if (page < 0 || page >= p.num_pages) {
          atomicOr(p.status, TLLM_FLAG_BAD_PAGE);
        } else {
          row = ((int64_t)page * p.Hkv + g) * p.bs + t % p.bs;
          ks = p.k_scales ? p.k_scales[row] : 1.f;
          vs = p.v_scales ? p.v_scales[row] : 1.f;
        }
      }
      row_s[tid] = row;
      ks_s[tid] = ks;
      vs_s[tid] = vs;
    }
    __syncthreads();
    for (int idx = tid; idx < kTile * D; idx += kThreads) {
      int j = idx / D, d = idx % D;
      int64_t row = row_s[j];
      float kv = 0.f, vv = 0.f;
      if (row >= 0) {
        kv = to_f32(kc[row * D + d]);
        // row = (page * Hkv + g) * bs + slot; a dimension-major V page keeps each
        // dimension's bs values together
        const int64_t slot = row % p.bs;
        vv = to_f32(vc[p.v_dim_major ? (row - slot) * D + (int64_t)d * p.bs + slot : row * D + d]);
      }
      k_s[j * (D + 1) + d] = kv;
      v_s[j * D + d] = vv;
    }
    __syncthreads();
    // Scores: lane = token, warp owns rows warp + 4k.
    {
      const int t = tt + lane;
      const bool tok_ok = row_s[lane] >= 0;
      for (int k = 0; k < kRows / 4; k++) {
        const int j = warp + 4 * k;
        float s = 0.f;
        const float* qr = q_s + j * D;
        const float* kr = k_s + lane * (D + 1);
#pragma unroll 8
        for (int d = 0; d < D; d++) s = fmaf(qr[d], kr[d], s);
        s *= ks_s[lane];
        const int pr = pos[k];
        const bool vis = tok_ok && pr >= 0 && t <= pr && (p.window <= 0 || pr - t < p.window);
        s = vis ? s : -INFINITY;
        float mx = s;
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_new = fmaxf(m_run[k], mx);
        float pv = 0.f, alpha = 1.f;
        if (m_new != -INFINITY) {
          pv = exp2f(s - m_new);
          alpha = exp2f(m_run[k] - m_new);
        }
        float sum = pv;
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        l_run[k] = l_run[k] * alpha + sum;
        m_run[k] = m_new;
        p_s[j * kTile + lane] = pv * vs_s[lane];
        if (lane == 0) alpha_s[j] = alpha;
      }
    }
    __syncthreads();
    // P.V: thread owns columns tid + 128c.
    for (int c = 0; c < DC; c++) {
      const int d = tid + c * kThreads;
      if (d >= D) break;
      for (int j = 0; j < kRows; j++) {
        float a = acc[j][c] * alpha_s[j];
        const float* pr = p_s + j * kTile;
#pragma unroll 8
        for (int t = 0; t < kTile; t++) a = fmaf(pr[t], v_s[t * D + d], a);
        acc[j][c] = a;
      }
    }
  }
  __syncthreads();
  if (lane == 0) {
    for (int k = 0; k < kRows / 4; k++) {
      m_s[warp + 4 * k] = m_run[k];
      l_s[warp + 4 * k] = l_run[k];
    }
  }
  __syncthreads();

  const int u_split = u * p.max_splits + split;
  for (int j = 0; j < kRows; j++) {
    const int r = r0 + j;
    if (r >= p.R) break;
    const float m = m_s[j], l = l_s[j];
    const int i = r / p.G, h = g * p.G + r % p.G;
    if (finalize) {
      float mul = 0.f;
      if (l > 0.f) {
        if (p.sinks) {
          const float sk = p.sinks[h] * kLog2e;
          const float M = fmaxf(m, sk);
          mul = exp2f(m - M) / (l * exp2f(m - M) + exp2f(sk - M));
        } else {
          mul = 1.f / l;
        }
      }
      const int64_t ob = ((int64_t)(b * p.Lq + i) * p.Hq + h) * D;
      for (int c = 0; c < DC; c++) {
        const int d = tid + c * kThreads;
        if (d < D) store_f32(p.out, p.out_dtype, ob + d, acc[j][c] * mul);
      }
    } else {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t o = ((int64_t)u_split * p.R + r) * D;
      for (int c = 0; c < DC; c++) {
        const int d = tid + c * kThreads;
        if (d < D) store_rec(p, o + d, acc[j][c] * inv);
      }
      if (tid == 0) p.ws_lse[(int64_t)u_split * p.R + r] = l > 0.f ? m + log2f(l) : -INFINITY;
    }
  }
}

template <int D>
constexpr size_t generic_smem_bytes() {
  return sizeof(float) * (kRows * D + kTile * (D + 1) + kTile * D + kRows * kTile + 2 * kTile + 3 * kRows + 2) +
         sizeof(int64_t) * kTile;
}

template <typename KT, int D>
cudaError_t launch_t(const Params& p, cudaStream_t stream) {
  auto kern = partial_generic_kernel<KT, D>;
  constexpr size_t smem = generic_smem_bytes<D>();
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.B * p.Hkv, p.num_splits, (p.R + kRows - 1) / kRows);
  kern<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <typename KT>
cudaError_t launch_d(const Params& p, cudaStream_t s) {
  switch (p.D) {
    case 64: return launch_t<KT, 64>(p, s);
    case 128: return launch_t<KT, 128>(p, s);
    case 256: return launch_t<KT, 256>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool generic_supports(const tllm_decode_attn_desc& d, int rows) {
  (void)rows;
  return d.head_dim == 64 || d.head_dim == 128 || d.head_dim == 256;
}

cudaError_t launch_partial_generic(const Params& p, cudaStream_t s) {
  switch (p.kv_dtype) {
    case TLLM_F16: return launch_d<__half>(p, s);
    case TLLM_BF16: return launch_d<__nv_bfloat16>(p, s);
    case TLLM_FP8_E4M3: return launch_d<e4m3_t>(p, s);
    case TLLM_INT8: return launch_d<i8_t>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace tllm
