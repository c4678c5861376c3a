// C ABI: planner, argument checks, workspace layout and launches.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"

using namespace tllm;

namespace {

constexpr size_t kHeaderBytes = 256;        // status word; the arrival counters follow

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Status word plus one arrival counter per (request, kv head) for the fused combine.
size_t header_bytes(int32_t batch, int32_t hkv) { return kHeaderBytes + align256((size_t)batch * hkv * 4); }

bool q_ok(int t) { return t == TLLM_F16 || t == TLLM_BF16 || t == TLLM_F32; }
bool kv_ok(int t) { return t == TLLM_F16 || t == TLLM_BF16 || t == TLLM_FP8_E4M3 || t == TLLM_INT8; }
bool quantised(int t) { return t == TLLM_FP8_E4M3 || t == TLLM_INT8; }

tllm_status check_desc(const tllm_decode_attn_desc* d) {
  if (!d) return TLLM_ERR_INVALID_ARG;
  if (d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->num_q_heads % d->num_kv_heads) return TLLM_ERR_INVALID_ARG;
  if (d->block_size <= 0 || d->max_blocks_per_seq <= 0 || d->num_pages <= 0) return TLLM_ERR_INVALID_ARG;
  if (d->head_dim <= 0 || !(d->softmax_scale >= 0.f) || !isfinite(d->softmax_scale)) return TLLM_ERR_INVALID_ARG;
  if ((int64_t)d->max_blocks_per_seq * d->block_size > (int64_t)1 << 30) return TLLM_ERR_INVALID_ARG;
  if (!q_ok(d->q_dtype) || !kv_ok(d->kv_dtype) || !q_ok(d->out_dtype)) return TLLM_ERR_UNSUPPORTED;
  if (d->block_size > 256) return TLLM_ERR_UNSUPPORTED;
  if (d->kernel < TLLM_KERNEL_AUTO || d->kernel > TLLM_KERNEL_TC_B16) return TLLM_ERR_INVALID_ARG;
  if (d->v_layout != TLLM_V_TOKEN_MAJOR && d->v_layout != TLLM_V_DIM_MAJOR) return TLLM_ERR_INVALID_ARG;
  if (d->record_type != TLLM_RECORD_F32 && d->record_type != TLLM_RECORD_BF16 && d->record_type != TLLM_RECORD_F16)
    return TLLM_ERR_INVALID_ARG;
  if (d->combine_mode != TLLM_COMBINE_KERNEL && d->combine_mode != TLLM_COMBINE_FUSED) return TLLM_ERR_INVALID_ARG;
  if (d->test_stall != 0 && d->test_stall != 1) return TLLM_ERR_INVALID_ARG;
  return TLLM_OK;
}

// Planning traits of a kernel variant: tokens per tile (split boundaries align to it),
// resident CTAs per SM, CTAs per (request, kv head, split), and the fixed cost of one CTA or
// item (set-up, pipeline fill, epilogue) expressed in tokens of streaming. persistent: CTAs
// take the items of the device work list in turn (item k to CTA k mod grid), so the plan can
// simulate each CTA's load. hbm_bound: one CTA alone streams faster than its share of HBM, so
// when some SMs run out of work the others speed up; its time then follows the work per SM
// (but no less than the longest item), not the number of waves. combine_tokens: the in-call
// cost of the combine launch that a plan with more than one split adds.
struct KernelTraits {
  int tile;
  int ctas_per_sm;
  int row_blocks;
  int overhead_tokens;
  bool hbm_bound = false;
  int combine_tokens = 0;
  bool persistent = false;
};

KernelTraits traits(int kernel, const tllm_decode_attn_desc& d, int rows) {

  switch (kernel) {
    case TLLM_KERNEL_TC_FP8: return KernelTraits{128, 1, 1, 1024, false, 512, true};
    case TLLM_KERNEL_SIMT: return KernelTraits{simt_tile(d.head_dim), 2, (rows + 7) / 8, 256};
    case TLLM_KERNEL_TC_I8: return KernelTraits{64, 1, 1, 512, false, 128, true};
    case TLLM_KERNEL_TC_B16: return KernelTraits{128, 1, 1, 256, true, 700};
    default: return KernelTraits{32, 2, (rows + 15) / 16, 64};
  }
}

// Busiest CTA of a persistent kernel, in tokens of streaming: the items of the work list
// (unit-major, each split's tiles plus the fixed cost of an item) dealt to `grid` CTAs in turn.
double persistent_cost(const std::vector<int>& ctx, int Lq, int window, int S, int min_chunk, int align, int Hkv,
                       int tile, double overhead, int grid, std::vector<double>& load) {
  load.assign(grid, 0.0);
  int64_t k = 0;
  for (int c : ctx) {
    const Span sp = request_span(c, Lq, window, S, min_chunk, align);
    for (int g = 0; g < Hkv; g++) {
      for (int s = 0; s < sp.nsplit; s++, k++) {
        const int t0 = sp.base + s * sp.chunk, t1 = std::min(c, t0 + sp.chunk);
        const int tiles = t1 > t0 ? (t1 - t0 + tile - 1) / tile : 0;
        load[k % grid] += (double)tiles * tile + overhead;
      }
    }
  }
  double mx = 0.0;
  for (double v : load) mx = std::max(mx, v);
  return mx;
}

bool kernel_supports(int kernel, const tllm_decode_attn_desc& d, int rows) {
  switch (kernel) {
    case TLLM_KERNEL_GENERIC: return generic_supports(d, rows);
    case TLLM_KERNEL_TC_FP8: return tc_fp8_supports(d, rows);
    case TLLM_KERNEL_SIMT: return simt_supports(d, rows);
    case TLLM_KERNEL_TC_I8: return tc_i8_supports(d, rows);
    case TLLM_KERNEL_TC_B16: return tc_b16_supports(d, rows);
    default: return false;
  }
}

int choose_kernel(const tllm_decode_attn_desc& d, int rows) {
  if (d.kernel != TLLM_KERNEL_AUTO) return d.kernel;
  if (tc_fp8_supports(d, rows)) return TLLM_KERNEL_TC_FP8;
  if (tc_b16_supports(d, rows)) return TLLM_KERNEL_TC_B16;
  if (tc_i8_supports(d, rows) && rows > 8) return TLLM_KERNEL_TC_I8;
  if (simt_supports(d, rows)) return TLLM_KERNEL_SIMT;
  if (tc_i8_supports(d, rows)) return TLLM_KERNEL_TC_I8;
  return TLLM_KERNEL_GENERIC;
}

int split_align(const KernelTraits& kt, int bs) {
  int a = kt.tile;
  if (bs > a) a = ((bs + kt.tile - 1) / kt.tile) * kt.tile;
  return a;
}

}  // namespace

namespace tllm {

int sm_count() {
  static std::atomic<int> cached[64];      // zero until first looked up (static storage)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

cudaError_t set_smem_attr(const void* func, int bytes) {
  struct Entry { const void* f; int dev; int bytes; };
  static Entry done[256];
  static int n_done = 0;
  static std::mutex mu;                    // launches may come from several host threads
  std::lock_guard<std::mutex> lock(mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < n_done; i++)
    if (done[i].f == func && done[i].dev == dev && done[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && n_done < 256) done[n_done++] = Entry{func, dev, bytes};
  return e;
}

}  // namespace tllm

extern "C" {

const char* tllm_status_string(tllm_status s) {
  switch (s) {
    case TLLM_OK: return "ok";
    case TLLM_ERR_INVALID_ARG: return "invalid argument";
    case TLLM_ERR_UNSUPPORTED: return "unsupported configuration";
    case TLLM_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case TLLM_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

tllm_status tllm_decode_attn_plan(const tllm_decode_attn_desc* desc, int32_t batch, int32_t query_len,
                                  int32_t window, const int32_t* host_ctx_lens, int64_t max_ctx_hint,
                                  int64_t total_ctx_hint, int32_t num_sms, int32_t splits_override,
                                  tllm_decode_attn_plan_t* out_plan) {
  tllm_status st = check_desc(desc);
  if (st != TLLM_OK) return st;
  if (!out_plan || batch <= 0 || query_len <= 0 || window < 0 || splits_override < 0) return TLLM_ERR_INVALID_ARG;
  const tllm_decode_attn_desc& d = *desc;
  const int G = d.num_q_heads / d.num_kv_heads;
  const int64_t rows64 = (int64_t)G * query_len;
  if (rows64 > 4096) return TLLM_ERR_UNSUPPORTED;
  const int rows = (int)rows64;
  const int kernel = choose_kernel(d, rows);
  if (!kernel_supports(kernel, d, rows)) return TLLM_ERR_UNSUPPORTED;
  const KernelTraits kt = traits(kernel, d, rows);
  const int max_ctx = d.max_blocks_per_seq * d.block_size;
  const int align = split_align(kt, d.block_size);
  const int min_chunk = align;                 // smallest split: one tile (or one page when pages are larger)
  if (num_sms <= 0) num_sms = 152;

  // Lengths the plan should fit: the host copy, else the hints (one request at the
  // longest context, the rest sharing the remaining total).
  std::vector<int> ctx;
  if (host_ctx_lens) {
    for (int b = 0; b < batch; b++) ctx.push_back(clamp_ctx(host_ctx_lens[b], max_ctx));
  } else {
    int64_t mx = max_ctx_hint > 0 ? std::min<int64_t>(max_ctx_hint, max_ctx) : max_ctx;
    int64_t tot = total_ctx_hint > 0 ? total_ctx_hint : mx * batch;
    ctx.push_back((int)mx);
    int64_t rest = std::max<int64_t>(0, tot - mx);
    for (int b = 1; b < batch; b++) ctx.push_back((int)std::min<int64_t>(mx, rest / (batch - 1)));
  }
  int max_vis = 0;
  for (int c : ctx) {
    Span s = request_span(c, query_len, window, 1, align, align);
    max_vis = std::max(max_vis, c - s.base);
  }
  const int s_cap = std::max(1, std::min(kMaxSplits, (max_vis + min_chunk - 1) / min_chunk));
  int S = 1;
  int chunk_floor = min_chunk;             // the plan's smallest split (tokens)
  if (splits_override > 0) {
    S = std::min(splits_override, kMaxSplits);
  } else if (kt.persistent) {
    // Work-based choice for the persistent kernels (aiter PR #5628, Changes: partitions sized
    // from the known KV work rather than a fixed CTA budget). A candidate is a split size c:
    // every request is cut into ceil(visible / c) splits of c tokens (S = the most any request
    // needs), and the work list deals the items to the CTAs in turn. Its estimated time is the
    // busiest CTA's load, plus the combine when any request splits. The candidates are the
    // even cuts of the longest request into s = 1 .. s_cap parts and the cuts that spread all
    // the work evenly over one to eight item waves. Ties go to fewer splits.
    const int slots = num_sms * kt.ctas_per_sm;
    int64_t total = 0;
    for (int c : ctx) total += (int64_t)(c - request_span(c, query_len, window, 1, align, align).base) * d.num_kv_heads;
    std::vector<int> cands;
    auto roundup = [&](int64_t x) { return (int)std::min<int64_t>(max_ctx, ((x + align - 1) / align) * align); };
    for (int s = 1; s <= s_cap; s++) cands.push_back(std::max(min_chunk, roundup((max_vis + s - 1) / s)));
    for (int w = 1; w <= 8; w++)
      cands.push_back(std::max(min_chunk, roundup((total + (int64_t)slots * w - 1) / ((int64_t)slots * w))));
    std::vector<std::pair<int, int>> options;        // (S, c)
    for (int c : cands) {
      int sc = 1;
      for (int x : ctx) {
        const int vis = x - request_span(x, query_len, window, 1, align, align).base;
        sc = std::max(sc, (vis + c - 1) / c);
      }
      options.emplace_back(std::min(sc, kMaxSplits), c);
    }
    std::sort(options.begin(), options.end());
    options.erase(std::unique(options.begin(), options.end()), options.end());
    std::vector<double> load;
    double best = 1e300;
    for (auto [sc, c] : options) {
      int64_t items = 0;
      for (int x : ctx) items += (int64_t)request_span(x, query_len, window, sc, c, align).nsplit * d.num_kv_heads;
      if (items > 32 * (int64_t)slots && sc > 1) continue;         // items too small for their fixed cost
      const int grid = (int)std::min<int64_t>((int64_t)batch * d.num_kv_heads * sc, slots);
      const double cost = persistent_cost(ctx, query_len, window, sc, c, align, d.num_kv_heads, kt.tile,
                                          kt.overhead_tokens, grid, load) +
                          (sc > 1 ? kt.combine_tokens : 0);
      if (cost < best * 0.999) {
        best = cost;
        S = sc;
        chunk_floor = c;
      }
    }
  } else {
    // Work-based choice: estimated time = waves x (chunk + per-CTA overhead), where a
    // wave is num_sms * ctas_per_sm CTAs; for an HBM-bound kernel, the tokens per slot (at
    // least the longest chunk) plus the overhead of its waves, plus the combine when split.
    // Ties go to fewer splits (less record traffic).
    const double slots = (double)num_sms * kt.ctas_per_sm;
    const double overhead = kt.overhead_tokens;
    double best = 1e300;
    for (int s = 1; s <= s_cap; s++) {
      int64_t ctas = 0, tokens = 0;
      int chunk = 0;
      for (int c : ctx) {
        Span sp = request_span(c, query_len, window, s, min_chunk, align);
        ctas += (int64_t)sp.nsplit * d.num_kv_heads * kt.row_blocks;
        tokens += (int64_t)(c - sp.base) * d.num_kv_heads * kt.row_blocks;
        chunk = std::max(chunk, sp.chunk);
      }
      double waves = ceil((double)ctas / slots);
      double cost = kt.hbm_bound ? std::max((double)tokens / slots, (double)chunk) + waves * overhead +
                                       (s > 1 ? kt.combine_tokens : 0)
                                 : waves * (chunk + overhead);
      if (cost < best * 0.999) {
        best = cost;
        S = s;
      }
    }
  }
  memset(out_plan, 0, sizeof(*out_plan));
  out_plan->desc = d;
  out_plan->desc.kernel = (tllm_kernel)kernel;
  out_plan->batch = batch;
  out_plan->query_len = query_len;
  out_plan->window = window;
  out_plan->num_splits = S;
  out_plan->max_splits = S;
  out_plan->min_chunk = chunk_floor;
  out_plan->split_align = align;
  out_plan->kernel = kernel;
  out_plan->rows = rows;
  const size_t units = (size_t)batch * d.num_kv_heads * S * rows;
  const size_t rec_bytes = d.record_type == TLLM_RECORD_F32 ? 4 : 2;
  out_plan->workspace_bytes = header_bytes(batch, d.num_kv_heads) + align256(units * sizeof(float)) +
                              align256(units * (size_t)d.head_dim * rec_bytes);
  // Fused combine, when asked for: the CTA that writes a request's last split record merges
  // them all, so no combine kernel is launched. Only where that merge is small next to the
  // call: the CUDA-core few-row kernel (one row block: at most 8 rows) with at most 128 KB of
  // records per request.
  out_plan->fused_combine = d.combine_mode == TLLM_COMBINE_FUSED && kernel == TLLM_KERNEL_SIMT && S > 1 && rows <= 8 &&
                            (size_t)S * rows * d.head_dim * rec_bytes <= ((size_t)128 << 10);
  return TLLM_OK;
}

tllm_status tllm_decode_attn_workspace_layout(const tllm_decode_attn_plan_t* plan, size_t* status_off,
                                              size_t* lse_off, size_t* o_off) {
  if (!plan) return TLLM_ERR_INVALID_ARG;
  const size_t units = (size_t)plan->batch * plan->desc.num_kv_heads * plan->max_splits * plan->rows;
  if (status_off) *status_off = 0;
  const size_t hb = header_bytes(plan->batch, plan->desc.num_kv_heads);
  if (lse_off) *lse_off = hb;
  if (o_off) *o_off = hb + align256(units * sizeof(float));
  return TLLM_OK;
}

tllm_status tllm_decode_attn_split_range(const tllm_decode_attn_plan_t* plan, int32_t ctx, int32_t query_len,
                                         int32_t window, int32_t num_splits, int32_t split, int32_t* t0,
                                         int32_t* t1, int32_t* nsplits) {
  if (!plan || !t0 || !t1 || query_len <= 0 || window < 0 || num_splits <= 0 || split < 0) return TLLM_ERR_INVALID_ARG;
  const int c = clamp_ctx(ctx, plan->desc.max_blocks_per_seq * plan->desc.block_size);
  Span sp = request_span(c, query_len, window, num_splits, plan->min_chunk, plan->split_align);
  if (nsplits) *nsplits = sp.nsplit;
  int a = sp.base + split * sp.chunk;
  int b = std::min(c, a + sp.chunk);
  if (split >= sp.nsplit) a = b = c;
  *t0 = a;
  *t1 = std::max(a, b);
  return TLLM_OK;
}

}  // extern "C"

namespace tllm {

// Checks the call arguments against the plan and, when they pass, fills the launch
// parameters. Queues nothing and makes no CUDA call.
tllm_status make_params(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                        const int32_t* context_lens, int32_t query_len, const float* kv_scales,
                        const float* sinks, int32_t window, int32_t num_splits, const tllm_workspace* ws,
                        void* out, Params* p) {
  if (!ws || !ws->plan || !ws->ptr) return TLLM_ERR_INVALID_ARG;
  const tllm_decode_attn_plan_t& pl = *ws->plan;
  tllm_status st = check_desc(&pl.desc);
  if (st != TLLM_OK) return st;
  const tllm_decode_attn_desc& d = pl.desc;
  if (!q || !k_cache || !v_cache || !context_lens || !out) return TLLM_ERR_INVALID_ARG;
  // no block table: a contiguous cache, request b's block i at page b * max_blocks_per_seq + i
  if (!block_table && (int64_t)pl.batch * d.max_blocks_per_seq > d.num_pages) return TLLM_ERR_INVALID_ARG;
  if (quantised(d.kv_dtype) && !kv_scales) return TLLM_ERR_INVALID_ARG;
  if (query_len <= 0 || query_len > pl.query_len || window < 0) return TLLM_ERR_INVALID_ARG;
  if (num_splits <= 0 || num_splits > pl.max_splits) return TLLM_ERR_INVALID_ARG;
  if (pl.batch <= 0 || pl.rows != (d.num_q_heads / d.num_kv_heads) * pl.query_len) return TLLM_ERR_INVALID_ARG;
  if (pl.split_align <= 0 || pl.min_chunk < pl.split_align) return TLLM_ERR_INVALID_ARG;
  if (ws->bytes < pl.workspace_bytes) return TLLM_ERR_WORKSPACE_TOO_SMALL;
  if (((uintptr_t)ws->ptr & 255) != 0) return TLLM_ERR_INVALID_ARG;
  if (!kernel_supports(pl.kernel, d, pl.rows)) return TLLM_ERR_UNSUPPORTED;
  size_t so, lo, oo;
  tllm_decode_attn_workspace_layout(&pl, &so, &lo, &oo);
  memset(p, 0, sizeof(*p));
  p->q = q;
  p->k_cache = k_cache;
  p->v_cache = v_cache;
  p->block_table = block_table;
  p->context_lens = context_lens;
  const size_t plane = (size_t)d.num_pages * d.num_kv_heads * d.block_size;
  p->k_scales = quantised(d.kv_dtype) ? kv_scales : nullptr;
  p->v_scales = quantised(d.kv_dtype) ? kv_scales + plane : nullptr;
  p->sinks = sinks;
  p->out = out;
  char* base = static_cast<char*>(ws->ptr);
  p->status = reinterpret_cast<uint32_t*>(base + so);
  p->counters = reinterpret_cast<uint32_t*>(base + kHeaderBytes);
  p->ws_lse = reinterpret_cast<float*>(base + lo);
  p->ws_o = reinterpret_cast<float*>(base + oo);
  p->B = pl.batch;
  p->Lq = query_len;
  p->Hq = d.num_q_heads;
  p->Hkv = d.num_kv_heads;
  p->G = d.num_q_heads / d.num_kv_heads;
  p->D = d.head_dim;
  p->R = p->G * query_len;
  p->bs = d.block_size;
  p->max_blocks = d.max_blocks_per_seq;
  p->num_pages = d.num_pages;
  p->window = window;
  p->num_splits = num_splits;
  p->max_splits = pl.max_splits;
  p->min_chunk = pl.min_chunk;
  p->align = pl.split_align;
  p->max_ctx = d.max_blocks_per_seq * d.block_size;
  const float scale = d.softmax_scale > 0.f ? d.softmax_scale : 1.f / sqrtf((float)d.head_dim);
  p->scale_log2 = scale * kLog2e;
  p->q_dtype = d.q_dtype;
  p->kv_dtype = d.kv_dtype;
  p->out_dtype = d.out_dtype;
  p->v_dim_major = d.v_layout == TLLM_V_DIM_MAJOR;
  p->rec_type = d.record_type;
  p->fused = pl.fused_combine != 0;
  p->test_stall = d.test_stall;
  // alignment the chosen kernel's copies need (TMA boxes, 16-byte loads and stores)
  bool aligned = true;
  switch (pl.kernel) {
    case TLLM_KERNEL_TC_FP8: aligned = tc_fp8_pointers_ok(*p); break;
    case TLLM_KERNEL_TC_I8: aligned = tc_i8_pointers_ok(*p); break;
    case TLLM_KERNEL_SIMT: aligned = simt_pointers_ok(*p); break;
    case TLLM_KERNEL_TC_B16: aligned = tc_b16_pointers_ok(*p); break;
    default: break;
  }
  return aligned ? TLLM_OK : TLLM_ERR_INVALID_ARG;
}

}  // namespace tllm

namespace {

tllm_status run_partial(const Params& p, int kernel, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidValue;
  // (make_params has checked the pointers' alignment for the kernel)
  switch (kernel) {
    case TLLM_KERNEL_GENERIC: e = launch_partial_generic(p, s); break;
    case TLLM_KERNEL_TC_FP8: e = launch_partial_tc_fp8(p, s); break;
    case TLLM_KERNEL_TC_I8: e = launch_partial_tc_i8(p, s); break;
    case TLLM_KERNEL_SIMT: e = launch_partial_simt(p, s); break;
    case TLLM_KERNEL_TC_B16: e = launch_partial_tc_b16(p, s); break;
    default: return TLLM_ERR_UNSUPPORTED;
  }
  return e == cudaSuccess ? TLLM_OK : TLLM_ERR_CUDA;
}

}  // namespace

extern "C" {

tllm_status tllm_decode_attn_partial(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, const int32_t* context_lens, int32_t query_len,
                                     const float* kv_scales, const float* sinks, int32_t window, int32_t num_splits,
                                     const tllm_workspace* workspace, void* out, tllm_stream_t stream) {
  Params p;
  tllm_status st = make_params(q, k_cache, v_cache, block_table, context_lens, query_len, kv_scales, sinks, window,
                               num_splits, workspace, out, &p);
  if (st != TLLM_OK) return st;
  return run_partial(p, workspace->plan->kernel, (cudaStream_t)stream);
}

tllm_status tllm_decode_attn_combine(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, const int32_t* context_lens, int32_t query_len,
                                     const float* kv_scales, const float* sinks, int32_t window, int32_t num_splits,
                                     const tllm_workspace* workspace, void* out, tllm_stream_t stream) {
  Params p;
  tllm_status st = make_params(q, k_cache, v_cache, block_table, context_lens, query_len, kv_scales, sinks, window,
                               num_splits, workspace, out, &p);
  if (st != TLLM_OK) return st;
  if (num_splits <= 1 || p.fused) return TLLM_OK;     // fused: the partial kernel merged
  return launch_combine(p, (cudaStream_t)stream) == cudaSuccess ? TLLM_OK : TLLM_ERR_CUDA;
}

tllm_status tllm_decode_attn_splitkv(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, const int32_t* context_lens, int32_t query_len,
                                     const float* kv_scales, const float* sinks, int32_t window, int32_t num_splits,
                                     const tllm_workspace* workspace, void* out, tllm_stream_t stream) {
  Params p;
  tllm_status st = make_params(q, k_cache, v_cache, block_table, context_lens, query_len, kv_scales, sinks, window,
                               num_splits, workspace, out, &p);
  if (st != TLLM_OK) return st;
  st = run_partial(p, workspace->plan->kernel, (cudaStream_t)stream);
  if (st != TLLM_OK || num_splits <= 1 || p.fused) return st;
  return launch_combine(p, (cudaStream_t)stream) == cudaSuccess ? TLLM_OK : TLLM_ERR_CUDA;
}

tllm_status tllm_decode_attn_read_status(const tllm_workspace* ws, uint32_t* flags, int32_t reset,
                                         tllm_stream_t stream) {
  if (!ws || !ws->ptr || !flags || ws->bytes < kHeaderBytes) return TLLM_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, ws->ptr, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return TLLM_ERR_CUDA;
  // reset: the status word, and with a plan the arrival counters of the fused combine too
  const size_t clear = ws->plan ? header_bytes(ws->plan->batch, ws->plan->desc.num_kv_heads) : sizeof(uint32_t);
  if (reset && cudaMemsetAsync(ws->ptr, 0, clear <= ws->bytes ? clear : sizeof(uint32_t), s) != cudaSuccess)
    return TLLM_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return TLLM_ERR_CUDA;
  *flags = v;
  return TLLM_OK;
}

}  // extern "C"
