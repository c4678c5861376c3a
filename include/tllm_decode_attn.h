/*
 * tllm_decode_attn.h -- C ABI of the GB300 (sm_103a) split-KV paged decode attention.
 *
 * The operation: for every request b, query row i < Lq and query head h,
 *
 *     out[b,i,h,:] = sum_t softmax_t( scale * q[b,i,h,:] . K_t [; sink_h] ) * V_t
 *
 * over the keys t the row may see (causal among the Lq rows, optionally a sliding
 * window), K_t / V_t read from a paged cache through a block table and dequantised
 * with per-token fp32 scales. The keys of each request are split into chunks that run
 * on separate CTAs; each chunk emits a normalised partial output and its log-sum-exp,
 * and a second kernel merges the chunks with a max-LSE-stabilised weighted sum.
 * Sources: "split-KV decode attention design record (TLLM-ATTN-SPLITKV)" (tiny-llm
 * PR #11), design section (partial grid over heads x splits, chunk = ceil(visible /
 * splits) computed on the device, flash-decoding combine, num_splits a host argument,
 * preallocated partials, new *_splitkv entry points); "split packed-Q8 verifier KV
 * scans" (hipfire PR #760), Summary (normalised O plus LSE records, stable max-LSE
 * merge); "[FlyDSL] perf(pa_decode): tune MTP work budgets and planned reduction"
 * (aiter PR #5628), Changes (work-based partition planning from host-known lengths,
 * a reducer that visits only each request's actual partitions, sliding window and
 * sinks, fixed capacity for graph replay).
 *
 * Conventions for every entry point:
 *   - The caller owns every buffer. Device pointers are plain CUDA device addresses
 *     on the current device; the library never allocates, frees or copies memory
 *     between host and device inside tllm_decode_attn_splitkv / _partial / _combine,
 *     never synchronises, and is therefore capturable in a CUDA graph.
 *   - Errors are returned as tllm_status before anything is launched; a launch
 *     failure reported by the CUDA runtime maps to TLLM_ERR_CUDA.
 *   - Bad DATA in device buffers (a context length beyond the block table, a page id
 *     outside the cache) never faults: the kernel clamps or masks it and sets a bit in
 *     the workspace status word (TLLM_FLAG_*), readable with tllm_decode_attn_read_status.
 *
 * Layouts (row-major, contiguous):
 *   q            [B, Lq, Hq, D]            q_dtype (f16, bf16 or f32)
 *   out          [B, Lq, Hq, D]            out_dtype (f16, bf16 or f32)
 *   k_cache      [num_pages, Hkv, bs, D]   kv_dtype (f16, bf16, fp8 e4m3 or int8)
 *   v_cache      [num_pages, Hkv, bs, D]   kv_dtype ([num_pages, Hkv, D, bs] with TLLM_V_DIM_MAJOR)
 *   kv_scales    [2, num_pages, Hkv, bs]   fp32: K scales then V scales (quantised KV only, else NULL)
 *   block_table  [B, max_blocks_per_seq]   int32 physical page ids, or NULL for a contiguous
 *                                          cache: block i of request b is then page
 *                                          b * max_blocks_per_seq + i (tiny-llm PR #11, design
 *                                          section: the ContiguousRows address mode)
 *   context_lens [B]                       int32 KV length INCLUDING the Lq new rows;
 *                                          row i sits at position ctx - Lq + i
 *   sinks        [Hq]                      fp32 sink logit per query head, or NULL
 *   Query head h uses KV head h / (Hq / Hkv).
 */
#ifndef TLLM_DECODE_ATTN_H
#define TLLM_DECODE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* tllm_stream_t;

typedef enum {
  TLLM_OK = 0,
  TLLM_ERR_INVALID_ARG = 1,          /* null pointer, bad size or a value outside the plan */
  TLLM_ERR_UNSUPPORTED = 2,          /* dtype / head_dim / block_size combination not built */
  TLLM_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace->bytes < plan->workspace_bytes */
  TLLM_ERR_CUDA = 4                  /* the CUDA runtime reported an error at launch */
} tllm_status;

typedef enum {
  TLLM_F16 = 0,
  TLLM_BF16 = 1,
  TLLM_F32 = 2,
  TLLM_FP8_E4M3 = 3,                 /* OCP e4m3 ("fn"), per-token fp32 scale */
  TLLM_INT8 = 4                      /* two's complement, per-token fp32 scale */
} tllm_dtype;

/* Partial-kernel variants. TLLM_KERNEL_AUTO lets the planner choose. */
typedef enum {
  TLLM_KERNEL_AUTO = 0,
  TLLM_KERNEL_GENERIC = 1,           /* CUDA-core kernel, every supported shape */
  TLLM_KERNEL_SIMT = 2,              /* pipelined CUDA-core kernel, 8 packed rows per CTA */
  TLLM_KERNEL_TC_FP8 = 3,            /* tcgen05 FP8 kernel, e4m3 KV, head_dim 128 */
  TLLM_KERNEL_TC_I8 = 4,             /* tcgen05 16-bit kernel, bf16 / f16 Q, <= 128 rows: int8 or e4m3 KV
                                        widened to f16, f16 / bf16 KV (head_dim 64 / 128 / 256; a
                                        16-bit cache at 256 with token-major V only) */
  TLLM_KERNEL_TC_B16 = 5             /* tcgen05 16-bit kernel, f16 / bf16 KV and Q, head_dim 128, <= 16 rows */
} tllm_kernel;

/* Layout of v_cache within a page (aiter PR #5628, Performance table: plain and "transposed"
 * V). K always uses the token-major layout. */
typedef enum {
  TLLM_V_TOKEN_MAJOR = 0,            /* v_cache [num_pages, Hkv, bs, D]: a token's D values contiguous */
  TLLM_V_DIM_MAJOR = 1               /* v_cache [num_pages, Hkv, D, bs]: each dimension's bs values contiguous
                                        (the transposed V cache) */
} tllm_v_layout;

/* Element type of the normalised partial outputs (split records) in the workspace. fp32 by
 * default; a 16-bit record halves the record traffic and the workspace (aiter PR #5628,
 * Changes: a 16-bit partial output per row plus fp32 scalars) at the cost of one rounding of
 * each partial output: 2^-9 relative for bf16, 2^-11 for f16 (whose range ends at 65504, so
 * f16 records suit caches whose dequantised values stay below that). The log-sum-exp stays fp32. */
typedef enum {
  TLLM_RECORD_F32 = 0,
  TLLM_RECORD_BF16 = 1,
  TLLM_RECORD_F16 = 2
} tllm_record_type;

/* How the split records are merged. TLLM_COMBINE_KERNEL: a combine kernel launched as a
 * programmatic dependent of the partial kernel, so its launch overlaps the partial's tail.
 * TLLM_COMBINE_FUSED: the partial CTA that writes a request's last record merges them all and
 * no combine kernel runs (tiny-llm PR #11, open question 1: the last CTA merges, an atomic
 * arrival ticket, no waiting); taken by the CUDA-core few-row kernel when a request's records
 * are at most 128 KB, else the plan keeps the combine kernel. On a GB300 the fused merge (a
 * GPU-wide fence, the ticket, then the records read by one CTA) measured about 2 us slower per
 * call than the overlapped kernel on the single-decode workload, hence the default. */
typedef enum {
  TLLM_COMBINE_KERNEL = 0,
  TLLM_COMBINE_FUSED = 1
} tllm_combine_mode;

/* Device status bits written into the workspace header. */
#define TLLM_FLAG_CTX_CLAMPED   0x1u  /* some context_lens[b] was < 0 or > max_blocks*bs; clamped */
#define TLLM_FLAG_BAD_PAGE      0x2u  /* some referenced page id was outside [0, num_pages); masked */
#define TLLM_FLAG_TIMEOUT       0x4u  /* a pipeline wait ran out of time; that call's output is invalid */

/* Static shape, fixed for the lifetime of a plan (and of a captured graph). */
typedef struct {
  int32_t num_q_heads;               /* Hq, a multiple of num_kv_heads */
  int32_t num_kv_heads;              /* Hkv */
  int32_t head_dim;                  /* D: 64, 128 or 256 */
  int32_t block_size;                /* bs: tokens per page, 1..256 */
  int32_t max_blocks_per_seq;        /* block_table row length */
  int32_t num_pages;                 /* pages in k_cache / v_cache */
  tllm_dtype q_dtype, kv_dtype, out_dtype;
  float softmax_scale;               /* 0 => 1/sqrt(head_dim) */
  tllm_kernel kernel;                /* TLLM_KERNEL_AUTO unless a test pins a variant */
  tllm_v_layout v_layout;            /* TLLM_V_TOKEN_MAJOR unless the V cache is transposed */
  tllm_record_type record_type;      /* TLLM_RECORD_F32 unless 16-bit split records are wanted */
  tllm_combine_mode combine_mode;    /* TLLM_COMBINE_KERNEL unless the fused merge is wanted */
  int32_t test_stall;                /* 0. 1 (failure-detection tests only): the widening tensor-core
                                        kernel's QK^T issuer issues nothing, so the pipeline's bounded
                                        waits run out; the call sets TLLM_FLAG_TIMEOUT and its output
                                        is not valid. Other kernels ignore it. */
} tllm_decode_attn_desc;

/* Host POD produced by tllm_decode_attn_plan; copy it freely. */
typedef struct {
  tllm_decode_attn_desc desc;
  int32_t batch;                     /* B: requests per call */
  int32_t query_len;                 /* Lq the plan (and the workspace) was sized for */
  int32_t window;                    /* sliding window the plan assumed, 0 = none */
  int32_t num_splits;                /* chosen S (the number of partitions per request) */
  int32_t max_splits;                /* capacity the workspace was sized for, >= num_splits */
  int32_t min_chunk;                 /* smallest split, in tokens, a multiple of split_align */
  int32_t split_align;               /* split boundaries sit on multiples of this many tokens */
  int32_t kernel;                    /* tllm_kernel chosen */
  int32_t rows;                      /* packed rows per (request, kv head) = (Hq/Hkv) * query_len */
  int32_t fused_combine;             /* 1: the partial kernel merges each request's splits itself
                                        and no combine kernel is launched (desc.combine_mode) */
  int32_t reserved[6];
  size_t workspace_bytes;            /* bytes the caller must provide */
} tllm_decode_attn_plan_t;

/* Caller-owned device workspace (256-byte aligned) plus the plan it was sized for. */
typedef struct {
  const tllm_decode_attn_plan_t* plan;
  void* ptr;
  size_t bytes;
} tllm_workspace;

/*
 * Plan a call shape (host only; no CUDA call).
 * Work-based split planning after aiter PR #5628 (Changes: partitions sized from
 * host-known KV work, explicit caps take precedence, windowed work capped by the
 * window union and tile alignment) and tiny-llm PR #11 (num_splits is a host
 * argument; the caller may fall back to one split).
 *   desc            static shape.
 *   batch           requests per call (B >= 1).
 *   query_len       query rows per request (Lq >= 1).
 *   window          sliding window in tokens, 0 = none.
 *   host_ctx_lens   optional [batch] host copy of the lengths the plan should fit;
 *                   NULL = use the hints.
 *   max_ctx_hint    longest context expected (used when host_ctx_lens is NULL;
 *                   <= 0 means max_blocks_per_seq * block_size).
 *   total_ctx_hint  sum of contexts expected (<= 0: batch * max_ctx_hint).
 *   num_sms         SMs to plan for (<= 0: 152).
 *   splits_override > 0 forces num_splits (capped at 256 and at what the longest
 *                   request can use); 0 = choose.
 *   out_plan        written on success.
 * Returns TLLM_OK, TLLM_ERR_INVALID_ARG or TLLM_ERR_UNSUPPORTED.
 */
tllm_status tllm_decode_attn_plan(const tllm_decode_attn_desc* desc, int32_t batch, int32_t query_len,
                                  int32_t window, const int32_t* host_ctx_lens, int64_t max_ctx_hint,
                                  int64_t total_ctx_hint, int32_t num_sms, int32_t splits_override,
                                  tllm_decode_attn_plan_t* out_plan);

/*
 * The whole operation: partial kernel, then (when num_splits > 1) the combine kernel,
 * on `stream`. tiny-llm PR #11, design section (new *_splitkv entry, partial +
 * flash-decoding combine, device-side lengths, zero allocation during capture).
 *   q, k_cache, v_cache, block_table, context_lens, kv_scales, sinks, out: device
 *     pointers in the layouts above (kv_scales required for FP8/INT8 KV, ignored
 *     otherwise; sinks may be NULL; block_table may be NULL for a contiguous cache, which
 *     then needs num_pages >= batch * max_blocks_per_seq). The tensor-core kernels also need q, k_cache,
 *     v_cache and kv_scales 16-byte aligned (TMA boxes, 16-byte query loads), and the
 *     FP8 and INT8 ones `out` too (16-byte row stores); a misaligned pointer returns
 *     TLLM_ERR_INVALID_ARG.
 *   query_len       <= plan->query_len.
 *   window          sliding window (0 = none); must equal plan->window when the plan
 *                   assumed a window, since splits were sized for it.
 *   num_splits      1 .. plan->max_splits.
 *   workspace       plan + device buffer of >= plan->workspace_bytes.
 * Returns TLLM_OK or an error status; nothing is launched on error.
 */
tllm_status tllm_decode_attn_splitkv(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, const int32_t* context_lens,
                                     int32_t query_len, const float* kv_scales, const float* sinks,
                                     int32_t window, int32_t num_splits, const tllm_workspace* workspace,
                                     void* out, tllm_stream_t stream);

/*
 * Stage 1 alone: the partial kernel. Requests with more than one split write their
 * per-split records (normalised O and LSE) into the workspace; requests that need
 * only one split are finalised directly into `out`. Same arguments as _splitkv.
 */
tllm_status tllm_decode_attn_partial(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, const int32_t* context_lens,
                                     int32_t query_len, const float* kv_scales, const float* sinks,
                                     int32_t window, int32_t num_splits, const tllm_workspace* workspace,
                                     void* out, tllm_stream_t stream);

/*
 * Stage 2 alone: merge the split records of every request with more than one split
 * (stable max-LSE reduction over the request's actual splits only, hipfire PR #760
 * Summary and aiter PR #5628 Changes), applying the sink once. Same arguments as
 * _splitkv; only context_lens, sinks, window, num_splits, workspace and out are read.
 */
tllm_status tllm_decode_attn_combine(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, const int32_t* context_lens,
                                     int32_t query_len, const float* kv_scales, const float* sinks,
                                     int32_t window, int32_t num_splits, const tllm_workspace* workspace,
                                     void* out, tllm_stream_t stream);

/*
 * Workspace layout of a plan (byte offsets from workspace->ptr), for callers that
 * inspect the split records:
 *   status  uint32 status word (TLLM_FLAG_*), at offset 0
 *           then, from byte 256 to lse, one uint32 arrival counter per (request, kv head) for
 *           the fused combine. The status word and the counters (the workspace header) must be
 *           zero before the first call; every call that completes leaves the counters at zero
 *           again. After a TLLM_FLAG_TIMEOUT they may not be: tllm_decode_attn_read_status with
 *           reset clears them.
 *   lse     fp32 [batch*Hkv][max_splits][rows], LSE of the split in log2 units
 *           (log2 sum_t 2^(s_t * log2 e)); -inf for a split with no visible key
 *   o       [batch*Hkv][max_splits][rows][head_dim], normalised partial output in the
 *           desc's record_type (fp32, bf16 or f16)
 * Row r of (request b, kv head g) is query row r / G of query head g*G + r % G.
 */
tllm_status tllm_decode_attn_workspace_layout(const tllm_decode_attn_plan_t* plan, size_t* status_off,
                                              size_t* lse_off, size_t* o_off);

/*
 * Key range [*t0, *t1) of split `split` of a request with context `ctx` (host copy of
 * the rule the kernels apply on the device). *nsplits receives how many splits the
 * request actually uses. Returns TLLM_ERR_INVALID_ARG on bad arguments.
 */
tllm_status tllm_decode_attn_split_range(const tllm_decode_attn_plan_t* plan, int32_t ctx, int32_t query_len,
                                         int32_t window, int32_t num_splits, int32_t split, int32_t* t0,
                                         int32_t* t1, int32_t* nsplits);

/*
 * Read (and optionally clear) the workspace status word; `reset` also zeroes the arrival
 * counters of the fused combine when workspace->plan is given. Synchronises `stream`;
 * do not call during graph capture.
 */
tllm_status tllm_decode_attn_read_status(const tllm_workspace* workspace, uint32_t* flags, int32_t reset,
                                         tllm_stream_t stream);

/* Static string for a status code. */
const char* tllm_status_string(tllm_status status);

/* Size of the library-owned record area used by tllm_decode_attn_splitkv_noalloc. */
#define TLLM_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * tllm_decode_attn_splitkv without a caller workspace. This entry point has no counterpart
 * in the papers; it exists for callers that cannot allocate device memory, for example
 * engines that reserve all device memory for their own pools, and plugin hosts that pass
 * kernels only their tensors.
 *   - The split records live in a library-owned device array of
 *     TLLM_NOALLOC_SCRATCH_BYTES bytes. Every GPU that loads the library holds that array
 *     until the process exits.
 *   - Arguments are those of tllm_decode_attn_splitkv, with `plan` in place of the
 *     workspace.
 *   - A plan whose workspace_bytes exceeds the array returns TLLM_ERR_WORKSPACE_TOO_SMALL,
 *     and nothing is launched.
 *   - Every argument is checked first; on any error nothing is queued on `stream`.
 *   - The call allocates and frees nothing. It zeroes the array's status word on `stream`,
 *     then runs the partial and combine kernels. tllm_decode_attn_noalloc_read_status reads
 *     that word afterwards.
 *   - All calls on a device share the one array, and it keeps the last call's contents.
 *     Calls that overlap on the GPU (unordered streams) race on it.
 *   - The first call on each device looks up the array's device address.
 */
tllm_status tllm_decode_attn_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                             const int32_t* block_table, const int32_t* context_lens,
                                             int32_t query_len, const float* kv_scales, const float* sinks,
                                             int32_t window, int32_t num_splits,
                                             const tllm_decode_attn_plan_t* plan, void* out,
                                             tllm_stream_t stream);

/*
 * The status word of the library-owned record area (TLLM_FLAG_*), the counterpart of
 * tllm_decode_attn_read_status for tllm_decode_attn_splitkv_noalloc: a TLLM_FLAG_TIMEOUT
 * here means the last no-alloc call's output is not valid. The next no-alloc call zeroes the
 * word again, so read it after the call whose result you check. `reset` non-zero clears it.
 * Synchronises `stream`; do not call during graph capture. No allocation.
 */
tllm_status tllm_decode_attn_noalloc_read_status(uint32_t* flags, int32_t reset, tllm_stream_t stream);

/* TLLM_NOALLOC_SCRATCH_BYTES as built into the library (for bindings that cannot read the macro). */
size_t tllm_decode_attn_noalloc_scratch_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* TLLM_DECODE_ATTN_H */
