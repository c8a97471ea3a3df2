// C ABI of libcb (declared in include/cb.h): argument and metadata
// validation, planning from the host mirrors, and the launch sequence of one
// step on the caller's stream.
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>

#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <unordered_map>

#include "cb.h"
#include "launch.h"
#include "plan.h"

namespace {

thread_local std::string g_message;
thread_local int g_cuda_error = 0;

cb_status fail(cb_status s, const std::string& msg) {
  g_message = msg;
  return s;
}

cb_status cuda_fail(cudaError_t e, const char* what) {
  g_cuda_error = (int)e;
  g_message = std::string(what) + ": " + cudaGetErrorString(e);
  return CB_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

cb_status check_dtype(int32_t dtype, int* elt) {
  if (dtype == CB_F32) { *elt = 4; return CB_OK; }
  if (dtype == CB_BF16) { *elt = 2; return CB_OK; }
  return fail(CB_ERR_INVALID_ARG, "dtype must be CB_F32 or CB_BF16");
}

}  // namespace

// Captured steps of one padded shape each: cudaGraphExec_t by key (every buffer
// pointer, every size, the padded counts and the KV-length bucket).
struct cb_graph_cache {
  int32_t q_interval = 1;
  int32_t kv_interval = 0;
  std::mutex mu;
  struct Entry {
    cudaGraphExec_t exec;
    long long launches[cb::kNumKernels];
  };
  std::unordered_map<std::string, Entry> graphs;
  long long captures = 0;
  long long replays = 0;
};

namespace {

template <typename T>
void put(std::string& k, const T& v) {
  k.append(reinterpret_cast<const char*>(&v), sizeof(v));
}

}  // namespace

namespace cb {

// Status reporting for entry points defined in other files of the library.
cb_status report_error(cb_status s, const char* msg) { return fail(s, msg); }
cb_status report_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }

}  // namespace cb

extern "C" {

const char* cb_status_string(int status) {
  switch (status) {
    case CB_OK: return "ok";
    case CB_ERR_INVALID_ARG: return "invalid argument";
    case CB_ERR_METADATA: return "inconsistent step metadata";
    case CB_ERR_UNSUPPORTED: return "unsupported shape";
    case CB_ERR_WORKSPACE: return "workspace missing or too small";
    case CB_ERR_CUDA: return "CUDA error";
    case CB_ERR_DEVICE_CHECK: return "device-side bounds check failed";
  }
  return "unknown status";
}

const char* cb_last_error_message(void) { return g_message.c_str(); }

int cb_last_cuda_error(void) { return g_cuda_error; }

int cb_abi_version(void) { return CB_ABI_VERSION; }

cb_status cb_write_kv(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                      const int64_t* slot_mapping, int32_t num_tokens, int32_t num_blocks,
                      int32_t block_size, int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                      int32_t* error_word, void* stream) {
  int elt = 0;
  cb_status st = check_dtype(dtype, &elt);
  if (st != CB_OK) return st;
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return fail(CB_ERR_INVALID_ARG, "sizes must be positive (num_tokens >= 0)");
  const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * elt;
  if (row_bytes % 16 != 0 || row_bytes > (1 << 30))
    return fail(CB_ERR_UNSUPPORTED, "Hkv * head_dim * element size must be a multiple of 16 bytes");
  if (num_tokens == 0) return CB_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping)
    return fail(CB_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(CB_ERR_INVALID_ARG, "K/V pointers must be 16-byte aligned");
  cudaError_t e = cb::launch_write_kv(k_new, v_new, k_cache, v_cache, slot_mapping, num_tokens,
                                      (int64_t)num_blocks * block_size, (int32_t)row_bytes,
                                      error_word, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "write_kv launch");
  return CB_OK;
}

cb_status cb_copy_blocks(const void* k_src, const void* v_src, void* k_dst, void* v_dst,
                         int64_t src_num_blocks, int64_t dst_num_blocks, const int32_t* src_ids,
                         const int32_t* dst_ids, int32_t n, int32_t block_size,
                         int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                         int32_t* error_word, void* stream) {
  int elt = 0;
  cb_status st = check_dtype(dtype, &elt);
  if (st != CB_OK) return st;
  if (n < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0 || block_size <= 0 ||
      num_kv_heads <= 0 || head_dim <= 0)
    return fail(CB_ERR_INVALID_ARG, "sizes must be positive (n >= 0)");
  const int64_t block_bytes = (int64_t)block_size * num_kv_heads * head_dim * elt;
  if (block_bytes % 16 != 0 || block_bytes / 16 > (int64_t)1 << 30)
    return fail(CB_ERR_UNSUPPORTED, "block_size * Hkv * head_dim * element size must be a multiple of 16 bytes");
  if (n == 0) return CB_OK;
  if (!k_src || !v_src || !k_dst || !v_dst || !src_ids || !dst_ids)
    return fail(CB_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(k_src) || !aligned16(v_src) || !aligned16(k_dst) || !aligned16(v_dst))
    return fail(CB_ERR_INVALID_ARG, "K/V pointers must be 16-byte aligned");
  cudaError_t e = cb::launch_copy_blocks(k_src, v_src, k_dst, v_dst, src_ids, dst_ids, n,
                                         src_num_blocks, dst_num_blocks, block_bytes, error_word,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
  return CB_OK;
}

size_t cb_workspace_size(int32_t num_requests, int32_t num_tokens, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim) {
  return cb::workspace_bytes(num_requests, num_tokens, num_q_heads, num_kv_heads, head_dim);
}

cb_status cb_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < cb::kWorkspaceHeaderBytes)
    return fail(CB_ERR_WORKSPACE, "workspace missing or smaller than its header");
  cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "workspace init");
  return CB_OK;
}

cb_status cb_read_error_word(void* workspace, int32_t* h_error, void* stream) {
  if (!workspace || !h_error) return fail(CB_ERR_INVALID_ARG, "null pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  *h_error = word;
  return word != 0 ? fail(CB_ERR_DEVICE_CHECK, "device bounds check recorded an error")
                   : CB_OK;
}

}  // extern "C"

namespace {

// The step for a plain block table (ring_blocks == 0) or a ring of recycled pages;
// with `graph`, captured once per padded shape and replayed.
cb_status paged_attention_impl(cb_graph_cache* graph, void* out, const void* q, void* k_cache,
                               void* v_cache,
                               const void* k_new, const void* v_new, const int64_t* slot_mapping,
                               const int32_t* query_start_loc, const int32_t* seq_lens,
                               const int32_t* block_table, int32_t block_table_stride,
                               int32_t ring_blocks, const int32_t* h_query_start_loc,
                               const int32_t* h_seq_lens, int32_t num_requests, int32_t num_tokens,
                               int32_t num_blocks, int32_t block_size, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, float scale,
                               int32_t sliding_window, int32_t dtype, uint32_t flags,
                               void* workspace, size_t workspace_bytes, void* stream) {
  // ---- arguments
  int elt = 0;
  cb_status st = check_dtype(dtype, &elt);
  if (st != CB_OK) return st;
  if (num_requests < 0 || num_tokens < 0)
    return fail(CB_ERR_INVALID_ARG, "num_requests and num_tokens must be >= 0");
  if (num_blocks <= 0 || block_size <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      head_dim <= 0 || block_table_stride < 0)
    return fail(CB_ERR_INVALID_ARG, "sizes must be positive");
  if (head_dim != 64 && head_dim != 128) return fail(CB_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (num_q_heads % num_kv_heads != 0)
    return fail(CB_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
  const int G = num_q_heads / num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
    return fail(CB_ERR_UNSUPPORTED, "num_q_heads / num_kv_heads must be 1, 2, 4, 8 or 16");
  if (!is_pow2(block_size) || block_size > 256)
    return fail(CB_ERR_UNSUPPORTED, "block_size must be a power of two <= 256");
  if (!h_query_start_loc || !h_seq_lens)
    return fail(CB_ERR_INVALID_ARG, "host mirrors of query_start_loc and seq_lens are required");
  if (!workspace || workspace_bytes < cb::workspace_bytes(num_requests, num_tokens, num_q_heads,
                                                          num_kv_heads, head_dim))
    return fail(CB_ERR_WORKSPACE, "workspace missing or smaller than cb_workspace_size()");
  if (!aligned16(workspace)) return fail(CB_ERR_INVALID_ARG, "workspace must be 16-byte aligned");

  // ---- host mirrors of the metadata
  if (h_query_start_loc[0] != 0) return fail(CB_ERR_METADATA, "query_start_loc[0] must be 0");
  int64_t max_pages = 0;
  for (int r = 0; r < num_requests; ++r) {
    const int32_t q_len = h_query_start_loc[r + 1] - h_query_start_loc[r];
    if (q_len < 0) return fail(CB_ERR_METADATA, "query_start_loc must be non-decreasing");
    if (q_len > h_seq_lens[r])
      return fail(CB_ERR_METADATA, "seq_lens[r] must be >= q_len of request r");
    const int64_t pages = ((int64_t)h_seq_lens[r] + block_size - 1) / block_size;
    if (pages > max_pages) max_pages = pages;
  }
  if (graph) {
    // padded shape: num_requests and num_tokens multiples of the query interval;
    // the tokens past query_start_loc[R] (and requests with q_len 0) are padding
    if (num_tokens % graph->q_interval != 0 || num_requests % graph->q_interval != 0)
      return fail(CB_ERR_INVALID_ARG,
                  "graph mode: num_requests and num_tokens must be multiples of q_interval");
    if (h_query_start_loc[num_requests] > num_tokens)
      return fail(CB_ERR_METADATA, "query_start_loc[R] must be <= num_tokens");
    if (stream == nullptr)
      return fail(CB_ERR_INVALID_ARG, "graph mode needs a created stream (not the legacy default)");
  } else if (h_query_start_loc[num_requests] != num_tokens) {
    return fail(CB_ERR_METADATA, "query_start_loc[R] must equal num_tokens");
  }
  if (ring_blocks > 0) {
    // every position the step reads or writes, from the first query's window start
    // to the last new token, must be live in the ring at once
    if (ring_blocks > block_table_stride)
      return fail(CB_ERR_METADATA, "block_table_stride is smaller than ring_blocks");
    for (int r = 0; r < num_requests; ++r) {
      const int32_t seq = h_seq_lens[r];
      if (seq <= 0) continue;
      const int32_t ctx = seq - (h_query_start_loc[r + 1] - h_query_start_loc[r]);
      const int32_t lo = ctx - sliding_window + 1 > 0 ? ctx - sliding_window + 1 : 0;
      if ((seq - 1) / block_size - lo / block_size + 1 > ring_blocks)
        return fail(CB_ERR_METADATA,
                    "ring_blocks too small for the window and this step's tokens of a request");
    }
  } else if (max_pages > block_table_stride) {
    return fail(CB_ERR_METADATA, "block_table_stride is smaller than ceil(seq_len / block_size)");
  }
  if (num_tokens == 0) return CB_OK;

  if (!out || !q || !k_cache || !v_cache || !query_start_loc || !seq_lens || !block_table)
    return fail(CB_ERR_INVALID_ARG, "null pointer");
  if (k_new && (!v_new || !slot_mapping))
    return fail(CB_ERR_INVALID_ARG, "k_new given without v_new or slot_mapping");
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(CB_ERR_INVALID_ARG, "q/out/cache pointers must be 16-byte aligned");

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* error_word = static_cast<int32_t*>(workspace);
  // 1. scatter the step's new K/V (the attention reads them back)
  auto scatter = [&]() -> cudaError_t {
    if (!k_new) return cudaSuccess;
    const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * elt;
    return cb::launch_write_kv(k_new, v_new, k_cache, v_cache, slot_mapping, num_tokens,
                               (int64_t)num_blocks * block_size, (int32_t)row_bytes, error_word, s);
  };

  // 2. attention
  cb::StepArgs a;
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.query_start_loc = query_start_loc;
  a.seq_lens = seq_lens;
  a.block_table = block_table;
  a.bt_stride = block_table_stride;
  a.ring_blocks = ring_blocks;
  a.num_requests = num_requests;
  a.num_tokens = num_tokens;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)head_dim);
  a.scale_log2 = sc * 1.4426950408889634f;
  a.sliding_window = sliding_window > 0 ? sliding_window : 0;
  a.dtype = dtype;
  a.test_expire_wait = (flags & CB_FLAG_TEST_WAIT_EXPIRY) ? 1 : 0;
  a.error_word = error_word;

  cb::Plan plan;
  if (!graph) {
    const cb::ScatterInputs rows{k_new, v_new, slot_mapping};
    cb::plan_step(plan, a, h_query_start_loc, h_seq_lens, flags, k_new ? &rows : nullptr,
                  workspace, workspace_bytes);
    cudaError_t e = plan.fused_scatter ? cudaSuccess : scatter();
    if (e != cudaSuccess) return cuda_fail(e, "write_kv launch");
    e = cb::run_plan(plan, a, s);
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    return CB_OK;
  }

  // ---- graph mode: every launch depends on the padded shape only
  // which kinds of rows the batch has: part of the key, so that a graph holds only
  // the launches its batches need
  bool has_decode = false, has_prefill = false;
  for (int r = 0; r < num_requests; ++r) {
    const int32_t ql = h_query_start_loc[r + 1] - h_query_start_loc[r];
    has_decode |= ql == 1 && h_seq_lens[r] > 0;
    has_prefill |= ql > 1;
  }
  if ((flags & CB_FLAG_PORTABLE_ONLY) ||
      !cb::plan_graph_step(plan, a, has_decode, has_prefill, workspace, workspace_bytes))
    return fail(CB_ERR_UNSUPPORTED,
                "graph mode covers bf16 steps that the split-KV decode and the tile prefill "
                "kernels both support");
  std::string key;
  for (const void* ptr : {(const void*)out, q, (const void*)k_cache, (const void*)v_cache, k_new,
                          v_new, (const void*)slot_mapping, (const void*)query_start_loc,
                          (const void*)seq_lens, (const void*)block_table, (const void*)workspace})
    put(key, ptr);
  for (int32_t v : {block_table_stride, num_requests, num_tokens, num_blocks, block_size,
                    num_q_heads, num_kv_heads, head_dim, a.sliding_window, dtype, (int32_t)flags})
    put(key, v);
  put(key, a.scale_log2);
  put(key, workspace_bytes);
  int64_t kv_bucket = 0;  // the longest sequence, padded to the KV interval
  if (graph->kv_interval > 0) {
    int32_t max_seq = 0;
    for (int r = 0; r < num_requests; ++r) max_seq = h_seq_lens[r] > max_seq ? h_seq_lens[r] : max_seq;
    kv_bucket = ((int64_t)max_seq + graph->kv_interval - 1) / graph->kv_interval;
  }
  put(key, kv_bucket);
  put(key, (int32_t)(has_decode ? 1 : 0) | (has_prefill ? 2 : 0));

  std::lock_guard<std::mutex> lock(graph->mu);
  auto it = graph->graphs.find(key);
  if (it == graph->graphs.end()) {
    cudaError_t e = cb::prepare_plan(plan, a);
    if (e != cudaSuccess) return cuda_fail(e, "graph kernel attributes");
    long long before[cb::kNumKernels], after[cb::kNumKernels];
    cb::launch_counts(before);
    const bool timing = cb::set_kernel_timing(false);  // no event nodes in the graph
    cudaGraph_t g = nullptr;
    cudaGraphExec_t exec = nullptr;
    e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
      e = scatter();
      if (e == cudaSuccess) e = cb::run_plan(plan, a, s);
      const cudaError_t e2 = cudaStreamEndCapture(s, &g);
      if (e == cudaSuccess) e = e2;
      if (e == cudaSuccess) e = cudaGraphInstantiate(&exec, g, 0);
      if (g) cudaGraphDestroy(g);
    }
    cb::set_kernel_timing(timing);
    cb::launch_counts(after);
    if (e != cudaSuccess) return cuda_fail(e, "graph capture");
    cb_graph_cache::Entry en;
    en.exec = exec;
    long long undo[cb::kNumKernels];
    for (int k = 0; k < cb::kNumKernels; ++k) {
      en.launches[k] = after[k] - before[k];
      undo[k] = -en.launches[k];  // captured, not run: counted when the graph runs
    }
    cb::note_replayed_launches(undo);
    it = graph->graphs.emplace(key, en).first;
    ++graph->captures;
  } else {
    ++graph->replays;
  }
  cudaError_t e = cudaGraphLaunch(it->second.exec, s);
  if (e != cudaSuccess) return cuda_fail(e, "graph launch");
  cb::note_replayed_launches(it->second.launches);
  return CB_OK;
}

}  // namespace

extern "C" {

cb_status cb_paged_attention(void* out, const void* q, void* k_cache, void* v_cache,
                             const void* k_new, const void* v_new, const int64_t* slot_mapping,
                             const int32_t* query_start_loc, const int32_t* seq_lens,
                             const int32_t* block_table, int32_t block_table_stride,
                             const int32_t* h_query_start_loc, const int32_t* h_seq_lens,
                             int32_t num_requests, int32_t num_tokens, int32_t num_blocks,
                             int32_t block_size, int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_dim, float scale, int32_t sliding_window, int32_t dtype,
                             uint32_t flags, void* workspace, size_t workspace_bytes,
                             void* stream) {
  return paged_attention_impl(nullptr, out, q, k_cache, v_cache, k_new, v_new, slot_mapping,
                              query_start_loc, seq_lens, block_table, block_table_stride, 0,
                              h_query_start_loc, h_seq_lens, num_requests, num_tokens, num_blocks,
                              block_size, num_q_heads, num_kv_heads, head_dim, scale,
                              sliding_window, dtype, flags, workspace, workspace_bytes, stream);
}

cb_status cb_paged_attention_ring(void* out, const void* q, void* k_cache, void* v_cache,
                                  const void* k_new, const void* v_new,
                                  const int64_t* slot_mapping, const int32_t* query_start_loc,
                                  const int32_t* seq_lens, const int32_t* block_table,
                                  int32_t block_table_stride, int32_t ring_blocks,
                                  const int32_t* h_query_start_loc, const int32_t* h_seq_lens,
                                  int32_t num_requests, int32_t num_tokens, int32_t num_blocks,
                                  int32_t block_size, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, float scale, int32_t sliding_window,
                                  int32_t dtype, uint32_t flags, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (ring_blocks <= 0) return fail(CB_ERR_INVALID_ARG, "ring_blocks must be positive");
  if (sliding_window <= 0)
    return fail(CB_ERR_INVALID_ARG, "a ring of recycled pages needs a sliding window");
  return paged_attention_impl(nullptr, out, q, k_cache, v_cache, k_new, v_new, slot_mapping,
                              query_start_loc, seq_lens, block_table, block_table_stride,
                              ring_blocks, h_query_start_loc, h_seq_lens, num_requests,
                              num_tokens, num_blocks, block_size, num_q_heads, num_kv_heads,
                              head_dim, scale, sliding_window, dtype, flags, workspace,
                              workspace_bytes, stream);
}

cb_status cb_graph_cache_create(int32_t q_interval, int32_t kv_interval, cb_graph_cache** cache) {
  if (!cache) return fail(CB_ERR_INVALID_ARG, "null pointer");
  *cache = nullptr;
  if (q_interval <= 0 || kv_interval < 0)
    return fail(CB_ERR_INVALID_ARG, "q_interval must be positive and kv_interval >= 0");
  cb_graph_cache* c = new (std::nothrow) cb_graph_cache();
  if (!c) return fail(CB_ERR_INVALID_ARG, "out of host memory");
  c->q_interval = q_interval;
  c->kv_interval = kv_interval;
  *cache = c;
  return CB_OK;
}

void cb_graph_cache_destroy(cb_graph_cache* cache) {
  if (!cache) return;
  for (auto& kv : cache->graphs) cudaGraphExecDestroy(kv.second.exec);
  delete cache;
}

cb_status cb_graph_cache_stats(cb_graph_cache* cache, int64_t* graphs, int64_t* captures,
                               int64_t* replays) {
  if (!cache) return fail(CB_ERR_INVALID_ARG, "null pointer");
  std::lock_guard<std::mutex> lock(cache->mu);
  if (graphs) *graphs = (int64_t)cache->graphs.size();
  if (captures) *captures = cache->captures;
  if (replays) *replays = cache->replays;
  return CB_OK;
}

cb_status cb_paged_attention_graphed(cb_graph_cache* cache, void* out, const void* q,
                                     void* k_cache, void* v_cache, const void* k_new,
                                     const void* v_new, const int64_t* slot_mapping,
                                     const int32_t* query_start_loc, const int32_t* seq_lens,
                                     const int32_t* block_table, int32_t block_table_stride,
                                     const int32_t* h_query_start_loc, const int32_t* h_seq_lens,
                                     int32_t num_requests, int32_t num_tokens, int32_t num_blocks,
                                     int32_t block_size, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, float scale, int32_t sliding_window,
                                     int32_t dtype, uint32_t flags, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  if (!cache) return fail(CB_ERR_INVALID_ARG, "null graph cache");
  return paged_attention_impl(cache, out, q, k_cache, v_cache, k_new, v_new, slot_mapping,
                              query_start_loc, seq_lens, block_table, block_table_stride, 0,
                              h_query_start_loc, h_seq_lens, num_requests, num_tokens, num_blocks,
                              block_size, num_q_heads, num_kv_heads, head_dim, scale,
                              sliding_window, dtype, flags, workspace, workspace_bytes, stream);
}

}  // extern "C"
