// tllm_decode_attn_splitkv_noalloc: the split-KV call for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc. Examples:
//   - serving engines that reserve all of device memory up front for their KV-cache pool
//     and hand kernels no allocator;
//   - plugin hosts that expose only the tensors of a call.
// Such callers still need somewhere to put the per-split partial records. This entry point
// keeps them in a file-scope device array of fixed size instead of a caller-provided
// workspace. The caller passes only the inputs and the output.
//
// Costs and rules:
//   - Every GPU that loads this library holds the array (TLLM_NOALLOC_SCRATCH_BYTES) until
//     the process exits.
//   - Every call on a device shares the one array, which keeps the last call's contents.
//     Calls whose work overlaps on the GPU (different streams, no ordering between them)
//     race on it; order them on one stream or with events.
//   - The first call on each device looks up the array's device address.
#include <mutex>

#include "common.cuh"

namespace {

// The records; never named by host code except through cudaGetSymbolAddress. In host
// code the symbol is only a stand-in for the device array, not a device address.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TLLM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per device.
tllm_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TLLM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return TLLM_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return TLLM_OK;
}

}  // namespace

extern "C" tllm_status tllm_decode_attn_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                        const int32_t* block_table, const int32_t* context_lens,
                                                        int32_t query_len, const float* kv_scales,
                                                        const float* sinks, int32_t window, int32_t num_splits,
                                                        const tllm_decode_attn_plan_t* plan, void* out,
                                                        tllm_stream_t stream) {
  if (!plan) return TLLM_ERR_INVALID_ARG;
  if (plan->workspace_bytes > (size_t)TLLM_NOALLOC_SCRATCH_BYTES) return TLLM_ERR_WORKSPACE_TOO_SMALL;
  // Every argument is checked before any CUDA call. make_params only does arithmetic on the
  // workspace address, so an aligned stand-in serves for the check.
  tllm_workspace ws;
  ws.plan = plan;
  ws.ptr = reinterpret_cast<void*>((uintptr_t)256);
  ws.bytes = TLLM_NOALLOC_SCRATCH_BYTES;
  tllm::Params params;
  tllm_status st = tllm::make_params(q, k_cache, v_cache, block_table, context_lens, query_len, kv_scales, sinks, window,
                               num_splits, &ws, out, &params);
  if (st != TLLM_OK) return st;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != TLLM_OK) return st;
  ws.ptr = scratch;
  // The header (status word and the fused combine's arrival counters) starts each call at zero.
  size_t lse_off = 0;
  tllm_decode_attn_workspace_layout(plan, nullptr, &lse_off, nullptr);
  if (cudaMemsetAsync(scratch, 0, lse_off, (cudaStream_t)stream) != cudaSuccess) return TLLM_ERR_CUDA;
  return tllm_decode_attn_splitkv(q, k_cache, v_cache, block_table, context_lens, query_len, kv_scales, sinks,
                                  window, num_splits, &ws, out, stream);
}

extern "C" tllm_status tllm_decode_attn_noalloc_read_status(uint32_t* flags, int32_t reset, tllm_stream_t stream) {
  if (!flags) return TLLM_ERR_INVALID_ARG;
  void* scratch = nullptr;
  tllm_status st = scratch_address(&scratch);
  if (st != TLLM_OK) return st;
  tllm_workspace ws;
  ws.plan = nullptr;
  ws.ptr = scratch;
  ws.bytes = TLLM_NOALLOC_SCRATCH_BYTES;
  return tllm_decode_attn_read_status(&ws, flags, reset, stream);
}

extern "C" size_t tllm_decode_attn_noalloc_scratch_bytes(void) { return (size_t)TLLM_NOALLOC_SCRATCH_BYTES; }
