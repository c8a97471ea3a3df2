// Batched block copy: for every pair i, block dst_ids[i] of the destination K/V
// caches becomes block src_ids[i] of the source caches. This is the data movement
// behind preemption by swapping and behind CPU offloading: a request's KV blocks
// are gathered into a staging buffer for one transfer to pinned host memory, and
// copied back into free pool blocks when it resumes ("Continuous batching
// mechanics", d9bl.com, section "Running out of KV cache memory"; "Continuous
// batching architecture", Transformers docs, section "Offloading"). Source and
// destination may be the same pool (a copy between pool blocks) or different
// buffers of the same block shape (pool <-> staging).
//
// A block is block_size * Hkv * D elements, contiguous in both caches (32 KB for
// bf16, block_size 16, Hkv 8, D 128). One CTA copies one block of one tensor with
// 16-byte vector loads, all issued before the stores: HBM-bound, a read and a
// write of each block, nothing else.
#include "common.cuh"
#include "launch.h"

namespace cb {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 8;

__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(const uint4* __restrict__ k_src, const uint4* __restrict__ v_src,
                   uint4* __restrict__ k_dst, uint4* __restrict__ v_dst,
                   const int32_t* __restrict__ src_ids, const int32_t* __restrict__ dst_ids,
                   int64_t src_blocks, int64_t dst_blocks, int32_t block_vecs,
                   int32_t* error_word) {
  grid_dependency_wait();  // the blocks may have been written by the previous kernel
  allow_dependent_launch();
  const int i = blockIdx.x;
  const int64_t s = src_ids[i];
  const int64_t d = dst_ids[i];
  if (s < 0 || s >= src_blocks || d < 0 || d >= dst_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) record_error(error_word, 0x1);
    return;
  }
  const uint4* src = (blockIdx.y == 0 ? k_src : v_src) + s * block_vecs;
  uint4* dst = (blockIdx.y == 0 ? k_dst : v_dst) + d * block_vecs;
  for (int base = 0; base < block_vecs; base += kCopyThreads * kCopyUnroll) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int j = base + u * kCopyThreads + threadIdx.x;
      if (j < block_vecs) v[u] = __ldg(src + j);
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int j = base + u * kCopyThreads + threadIdx.x;
      if (j < block_vecs) dst[j] = v[u];
    }
  }
}

cudaError_t launch_copy_blocks(const void* k_src, const void* v_src, void* k_dst, void* v_dst,
                               const int32_t* src_ids, const int32_t* dst_ids, int32_t n,
                               int64_t src_blocks, int64_t dst_blocks, int64_t block_bytes,
                               int32_t* error_word, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(kCopyBlocks, copy_blocks_kernel, dim3(n, 2), dim3(kCopyThreads), 0, stream,
                    static_cast<const uint4*>(k_src), static_cast<const uint4*>(v_src),
                    static_cast<uint4*>(k_dst), static_cast<uint4*>(v_dst), src_ids, dst_ids,
                    src_blocks, dst_blocks, (int32_t)(block_bytes / 16), error_word);
}

}  // namespace cb
