// Internal launchers (host side) of the libcb kernels. Not part of the C ABI.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace cb {

struct StepArgs {
  void* out;
  const void* q;
  void* k_cache;
  void* v_cache;
  const int32_t* query_start_loc;
  const int32_t* seq_lens;
  const int32_t* block_table;
  int32_t bt_stride;
  int32_t ring_blocks;  // 0: plain block table; > 0: logical block b at entry b % ring_blocks
  int32_t num_requests;
  int32_t num_tokens;
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  float scale_log2;  // softmax scale * log2(e)
  int32_t sliding_window;
  int32_t dtype;     // cb_dtype
  int32_t test_expire_wait;  // CB_FLAG_TEST_WAIT_EXPIRY: a consumer's first wait runs out
  int32_t* error_word;
};

enum KernelId {
  kWriteKv = 0,
  kPortableAttention = 1,
  kDecodeSplit = 2,
  kPrefillTc = 3,
  kCopyBlocks = 4,
  kDecodeCombine = 5,
  kNumKernels = 6
};

void note_launch_begin(KernelId id, cudaStream_t stream);
void note_launch_end(KernelId id, cudaStream_t stream);
// Launch accounting for CUDA-graph replays (a replay launches what the capture recorded).
void note_replayed_launches(const long long* per_kernel);
void launch_counts(long long* per_kernel);
// Per-kernel event timing of the calling thread on/off; returns the previous state.
bool set_kernel_timing(bool enable);

// Launch with the programmatic-stream-serialization attribute (the kernel may
// start while the previous one on the stream drains; it waits on the device).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(KernelId id, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  note_launch_begin(id, stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  note_launch_end(id, stream);
  return e;
}


cudaError_t launch_write_kv(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                            const int64_t* slot_mapping, int32_t num_tokens, int64_t num_slots,
                            int32_t row_bytes, int32_t* error_word, cudaStream_t stream);

// Block k_dst/v_dst[dst_ids[i]] = block k_src/v_src[src_ids[i]] for i < n (device ids).
cudaError_t launch_copy_blocks(const void* k_src, const void* v_src, void* k_dst, void* v_dst,
                               const int32_t* src_ids, const int32_t* dst_ids, int32_t n,
                               int64_t src_blocks, int64_t dst_blocks, int64_t block_bytes,
                               int32_t* error_word, cudaStream_t stream);

// Portable CUDA-core attention over the query rows of the requests listed in
// `rows_of` (all rows when mode == 0, only rows of requests with q_len == 1
// when mode == 1, only q_len > 1 when mode == 2).
cudaError_t launch_portable_attention(const StepArgs& a, int mode, cudaStream_t stream);

}  // namespace cb
