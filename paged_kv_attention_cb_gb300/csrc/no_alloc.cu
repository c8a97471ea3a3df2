// cb_paged_attention_no_alloc: the step of cb_paged_attention for callers
// that may not allocate device memory when they call the library -- for
// instance a plugin running inside a host program that owns the device memory
// pool and forbids allocations on its inference path, or a latency-critical
// caller that cannot afford the implicit device synchronisation of
// cudaMalloc/cudaFree. The scratch the step needs (device error word and
// split-KV partial results) lives in a
// fixed-size device array compiled into this library instead of a
// caller-provided workspace; the caller still passes every input and output.
#include <cuda_runtime.h>

#include <mutex>

#include "cb.h"
#include "plan.h"

namespace cb {
cb_status report_error(cb_status s, const char* msg);
cb_status report_cuda_error(cudaError_t e, const char* what);
}  // namespace cb

namespace {

// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kScratchBytes = CB_NO_ALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// In host code g_scratch names a host-side stand-in, not device memory: the
// device address is looked up once per device (with that device current) and
// cached here.
constexpr int kMaxDevices = 128;
void* g_scratch_dev[kMaxDevices] = {};
std::mutex g_scratch_mutex;

cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_dev[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" cb_status cb_paged_attention_no_alloc(
    void* out, const void* q, void* k_cache, void* v_cache, const void* k_new, const void* v_new,
    const int64_t* slot_mapping, const int32_t* query_start_loc, const int32_t* seq_lens,
    const int32_t* block_table, int32_t block_table_stride, const int32_t* h_query_start_loc,
    const int32_t* h_seq_lens, int32_t num_requests, int32_t num_tokens, int32_t num_blocks,
    int32_t block_size, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale,
    int32_t sliding_window, int32_t dtype, uint32_t flags, void* stream) {
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return cb::report_cuda_error(e, "no-alloc scratch address");

  // The workspace size cb_paged_attention checks for is an upper bound over
  // all plans; the plan of this call touches only its leading extent, which
  // must fit in the fixed array.
  const size_t bound = cb_workspace_size(num_requests, num_tokens, num_q_heads, num_kv_heads,
                                         head_dim);
  // sizes the planner divides by or indexes with are checked first; anything else
  // malformed is left to cb_paged_attention's validation, which reports it
  const bool plannable = h_query_start_loc != nullptr && h_seq_lens != nullptr &&
                         num_requests >= 0 && num_blocks > 0 && block_size > 0 &&
                         (block_size & (block_size - 1)) == 0 && block_size <= 256 &&
                         num_q_heads > 0 && num_kv_heads > 0 &&
                         num_q_heads % num_kv_heads == 0 && (head_dim == 64 || head_dim == 128);
  cb::StepArgs a = {};
  a.num_requests = num_requests;
  a.num_tokens = num_tokens;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.sliding_window = sliding_window > 0 ? sliding_window : 0;
  a.dtype = dtype;
  size_t extent = cb::kWorkspaceHeaderBytes;
  size_t zeroed = cb::kWorkspaceHeaderBytes;
  if (plannable) {
    cb::Plan plan;
    const cb::ScatterInputs rows{k_new, v_new, slot_mapping};
    cb::plan_step(plan, a, h_query_start_loc, h_seq_lens, flags, k_new ? &rows : nullptr, scratch,
                  bound);
    extent = cb::workspace_extent(plan, a);
    zeroed = cb::workspace_zeroed_prefix(a, bound);
  }
  if (extent > kScratchBytes || zeroed > kScratchBytes)
    return cb::report_error(CB_ERR_WORKSPACE,
                            "step needs more scratch than the allocation-free entry point's fixed "
                            "array (CB_NO_ALLOC_SCRATCH_BYTES); use cb_paged_attention with a "
                            "workspace");

  // the error word starts at zero on every call
  e = cudaMemsetAsync(scratch, 0, zeroed, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cb::report_cuda_error(e, "no-alloc scratch clear");
  return cb_paged_attention(out, q, k_cache, v_cache, k_new, v_new, slot_mapping, query_start_loc,
                            seq_lens, block_table, block_table_stride, h_query_start_loc,
                            h_seq_lens, num_requests, num_tokens, num_blocks, block_size,
                            num_q_heads, num_kv_heads, head_dim, scale, sliding_window, dtype,
                            flags, scratch, bound, stream);
}

extern "C" cb_status cb_no_alloc_read_error_word(int32_t* h_error, void* stream) {
  if (!h_error) return cb::report_error(CB_ERR_INVALID_ARG, "null pointer");
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return cb::report_cuda_error(e, "no-alloc scratch address");
  return cb_read_error_word(scratch, h_error, stream);
}
