// Portable CUDA-core paged attention (any query length; fp32 and bf16).
//
// The fp32 dtype specialisation of the step, and the path for shapes outside
// the tensor-core kernels' set (block_size below their tile granularity). One
// warp owns one (query row, KV head) pair and the G query heads that share the
// KV head: it walks the row's attended positions in logical order, resolves
// each through the block table ("Continuous Batching", languisher.top,
// section "Extension: the vLLM v1 implementation": logical_block = kv_pos /
// BLOCK_SIZE, physical_block = block_table[req][logical_block], offset kv_pos %
// BLOCK_SIZE) and keeps a running (max, sum, output) online softmax in fp32.
// The mask is only the bounds [lo, context_len + local_q] (same section).
//
// Lanes split the head dimension, so each K/V row is read as one coalesced
// D-element vector; dot products are finished with warp shuffles.
#include <float.h>

#include "common.cuh"
#include "launch.h"

namespace cb {

constexpr int kPortableWarps = 4;

template <typename T, int VPT>
CB_DEV void load_row(const T* p, float (&x)[VPT]) {
#pragma unroll
  for (int v = 0; v < VPT; ++v) x[v] = Elt<T>::to_f(p[v]);
}

template <typename T, int VPT, int G>
__global__ void __launch_bounds__(kPortableWarps * 32)
portable_attention_kernel(StepArgs a, int mode) {
  grid_dependency_wait();
  allow_dependent_launch();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t item = (int64_t)blockIdx.x * kPortableWarps + warp;
  const int Hkv = a.num_kv_heads;
  if (item >= (int64_t)a.num_tokens * Hkv) return;
  const int t = (int)(item / Hkv);
  const int g = (int)(item % Hkv);

  // Request of row t: the r with query_start_loc[r] <= t < query_start_loc[r + 1].
  int lo_r = 0, hi_r = a.num_requests;  // invariant: qsl[lo_r] <= t < qsl[hi_r]
  while (hi_r - lo_r > 1) {
    const int mid = (lo_r + hi_r) >> 1;
    if (__ldg(a.query_start_loc + mid) <= t) lo_r = mid; else hi_r = mid;
  }
  const int r = lo_r;
  const int q_start = __ldg(a.query_start_loc + r);
  const int q_len = __ldg(a.query_start_loc + r + 1) - q_start;
  if (mode == 1 && q_len != 1) return;
  if (mode == 2 && q_len == 1) return;
  const int context_len = __ldg(a.seq_lens + r) - q_len;
  const int max_kv_pos = context_len + (t - q_start);
  const int min_kv_pos = a.sliding_window > 0 ? max(0, max_kv_pos - a.sliding_window + 1) : 0;

  const int D = VPT * 32;
  const T* q = static_cast<const T*>(a.q) + ((int64_t)t * a.num_q_heads + g * G) * D + lane * VPT;
  float qv[G][VPT];
#pragma unroll
  for (int h = 0; h < G; ++h) load_row<T, VPT>(q + h * D, qv[h]);

  float m[G], l[G], o[G][VPT];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -FLT_MAX;
    l[h] = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) o[h][v] = 0.f;
  }

  const T* kc = static_cast<const T*>(a.k_cache);
  const T* vc = static_cast<const T*>(a.v_cache);
  const int32_t* bt = a.block_table + (int64_t)r * a.bt_stride;
  for (int p = min_kv_pos; p <= max_kv_pos; ++p) {
    const int blk = __ldg(bt + bt_entry(p / a.block_size, a.ring_blocks));
    if (blk < 0 || blk >= a.num_blocks) {
      if (lane == 0) record_error(a.error_word, 0x1);
      continue;
    }
    const int64_t row = ((int64_t)blk * a.block_size + p % a.block_size) * Hkv + g;
    float kv[VPT], vv[VPT];
    load_row<T, VPT>(kc + row * D + lane * VPT, kv);
    load_row<T, VPT>(vc + row * D + lane * VPT, vv);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float s = 0.f;
#pragma unroll
      for (int v = 0; v < VPT; ++v) s = fmaf(qv[h][v], kv[v], s);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      s *= a.scale_log2;
      const float m_new = fmaxf(m[h], s);
      const float alpha = exp2f(m[h] - m_new);
      const float pe = exp2f(s - m_new);
      l[h] = l[h] * alpha + pe;
#pragma unroll
      for (int v = 0; v < VPT; ++v) o[h][v] = fmaf(o[h][v], alpha, pe * vv[v]);
      m[h] = m_new;
    }
  }

  T* out = static_cast<T*>(a.out) + ((int64_t)t * a.num_q_heads + g * G) * D + lane * VPT;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) out[h * D + v] = Elt<T>::from_f(o[h][v] * inv);
  }
}

template <typename T, int VPT>
static cudaError_t launch_g(const StepArgs& a, int mode, cudaStream_t s, dim3 grid, dim3 block) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_pdl(kPortableAttention, portable_attention_kernel<T, VPT, 1>, grid, block, 0, s, a, mode);
    case 2: return launch_pdl(kPortableAttention, portable_attention_kernel<T, VPT, 2>, grid, block, 0, s, a, mode);
    case 4: return launch_pdl(kPortableAttention, portable_attention_kernel<T, VPT, 4>, grid, block, 0, s, a, mode);
    case 8: return launch_pdl(kPortableAttention, portable_attention_kernel<T, VPT, 8>, grid, block, 0, s, a, mode);
    case 16: return launch_pdl(kPortableAttention, portable_attention_kernel<T, VPT, 16>, grid, block, 0, s, a, mode);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_portable_attention(const StepArgs& a, int mode, cudaStream_t stream) {
  const int64_t items = (int64_t)a.num_tokens * a.num_kv_heads;
  if (items == 0) return cudaSuccess;
  const dim3 grid((unsigned)((items + kPortableWarps - 1) / kPortableWarps));
  const dim3 block(kPortableWarps * 32);
  const bool bf16 = a.dtype == 1;
  if (a.head_dim == 64)
    return bf16 ? launch_g<__nv_bfloat16, 2>(a, mode, stream, grid, block)
                : launch_g<float, 2>(a, mode, stream, grid, block);
  if (a.head_dim == 128)
    return bf16 ? launch_g<__nv_bfloat16, 4>(a, mode, stream, grid, block)
                : launch_g<float, 4>(a, mode, stream, grid, block);
  return cudaErrorInvalidValue;
}

}  // namespace cb
