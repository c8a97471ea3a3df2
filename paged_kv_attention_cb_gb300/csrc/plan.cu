// Host-side planning of one step from the host mirrors of the metadata. The
// scheduler metadata "already divides the work into a request's query tile /
// KV tile" ("Continuous Batching", languisher.top, section "Extension: the
// vLLM v1 implementation"); here that division is made per call.
#include "cb.h"
#include "plan.h"

namespace cb {

size_t workspace_bytes(int32_t num_requests, int32_t num_tokens, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim) {
  (void)num_tokens;
  (void)num_kv_heads;
  if (num_requests < 0 || num_q_heads <= 0 || head_dim <= 0) return kWorkspaceHeaderBytes;
  const size_t segments = (size_t)num_requests + kMaxDecodeCtas;
  const size_t partial = (size_t)num_q_heads * (head_dim + 2) * sizeof(float);
  return kWorkspaceHeaderBytes + segments * partial;
}

void plan_step(Plan& plan, const StepArgs& a, const int32_t* h_qsl, const int32_t* h_seq_lens,
               uint32_t flags, void* workspace, size_t workspace_bytes) {
  (void)h_qsl;
  (void)h_seq_lens;
  plan.workspace = workspace;
  plan.workspace_bytes = workspace_bytes;
  plan.fast_decode = false;
  plan.fast_prefill = false;
  plan.portable_mode = 0;
  if ((flags & CB_FLAG_PORTABLE_ONLY) || a.dtype == CB_F32) return;
}

cudaError_t run_plan(const Plan& plan, const StepArgs& a, cudaStream_t stream) {
  if (plan.portable_mode >= 0) {
    cudaError_t e = launch_portable_attention(a, plan.portable_mode, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace cb
