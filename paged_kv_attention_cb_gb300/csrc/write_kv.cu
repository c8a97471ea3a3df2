// KV scatter: the step's new K/V rows go to the flat cache slots named by
// slot_mapping ("Continuous Batching", languisher.top, section "Extension: the
// vLLM v1 implementation", where the scheduler builds slot_mapping).
//
// One token row is Hkv * D elements (2 KB for bf16, Hkv 8, D 128), contiguous
// both in k_new and in the cache slot, so each CTA copies whole rows with
// 16-byte vector loads and stores: a read and a write of the row, nothing
// else. HBM-bound: 2 * 2 * T * row_bytes moved per step.
#include "common.cuh"
#include "launch.h"

namespace cb {

// grid.x covers tokens (TOK_PER_CTA per CTA), blockDim.x = 128. The K row and
// the V row of a token are copied by the same threads.
constexpr int kScatterThreads = 128;

__global__ void __launch_bounds__(kScatterThreads)
write_kv_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                const int64_t* __restrict__ slot_mapping, int32_t num_tokens, int64_t num_slots,
                int32_t row_vecs, int32_t tok_per_cta, int32_t* error_word) {
  grid_dependency_wait();
  allow_dependent_launch();
  const int t0 = blockIdx.x * tok_per_cta;
  const int t1 = min(num_tokens, t0 + tok_per_cta);
  for (int t = t0; t < t1; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (threadIdx.x == 0) record_error(error_word, 0x2);
      continue;
    }
    const uint4* ks = k_new + (int64_t)t * row_vecs;
    const uint4* vs = v_new + (int64_t)t * row_vecs;
    uint4* kd = k_cache + slot * row_vecs;
    uint4* vd = v_cache + slot * row_vecs;
    for (int i = threadIdx.x; i < row_vecs; i += kScatterThreads) {
      const uint4 kv = __ldg(ks + i);
      const uint4 vv = __ldg(vs + i);
      kd[i] = kv;
      vd[i] = vv;
    }
  }
}

cudaError_t launch_write_kv(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                            const int64_t* slot_mapping, int32_t num_tokens, int64_t num_slots,
                            int32_t row_bytes, int32_t* error_word, cudaStream_t stream) {
  if (num_tokens <= 0) return cudaSuccess;
  const int row_vecs = row_bytes / 16;
  // Enough rows per CTA that a CTA moves >= ~4 KB per row pair, but keep the
  // grid at least a few CTAs per SM for small steps.
  const int tok_per_cta = row_vecs >= kScatterThreads ? 1 : 2;
  const int grid = (num_tokens + tok_per_cta - 1) / tok_per_cta;
  // Prefer the shared-memory-heavy carveout the attention kernels that follow
  // use, so the SMs are not reconfigured between the two launches.
  static bool carveout_set = false;
  if (!carveout_set) {
    cudaFuncSetAttribute(write_kv_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                         cudaSharedmemCarveoutMaxShared);
    carveout_set = true;
  }
  return launch_pdl(kWriteKv, write_kv_kernel, dim3(grid), dim3(kScatterThreads), 0, stream,
                    static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                    static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slot_mapping,
                    num_tokens, num_slots, row_vecs, tok_per_cta, error_word);
}

}  // namespace cb
