/*
 * cb.h -- C ABI of libcb, the GB300 (sm_103a) hot path of one continuous-batching
 * attention step over a paged KV cache.
 *
 * What it computes. A step packs the new query tokens of R requests into one
 * ragged stream ("Continuous Batching", languisher.top, section "Continuous
 * Batching": ragged batching). Request r owns query rows
 * [query_start_loc[r], query_start_loc[r+1]) and has seq_lens[r] KV positions
 * in total, the last q_len of which are this step's tokens, so its context is
 * context_len = seq_lens[r] - q_len. Query row local_q of request r attends KV
 * positions 0 .. context_len + local_q (the block-diagonal causal mask of the
 * section "Attention Mask construction", expressed only as these bounds, as in
 * the section "Extension: the vLLM v1 implementation"), optionally limited to
 * the last sliding_window of them. Logical position p of request r lives in
 * physical page block_table[r * stride + p / block_size] at offset
 * p % block_size (same section). The step's new K/V are first written to the
 * flat slots given by slot_mapping (same section, where the scheduler builds
 * slot_mapping, seq_lens, query_start_loc and block_table).
 *
 * Layouts (row-major, all tensors contiguous):
 *   q, out                 [T, Hq, D]           dtype (out has the dtype of q)
 *   k_new, v_new           [T, Hkv, D]          dtype
 *   k_cache, v_cache       [num_blocks, block_size, Hkv, D]   dtype
 *   slot_mapping           [T]       int64      flat slot = page * block_size + offset; < 0 skips
 *   query_start_loc        [R + 1]   int32      query_start_loc[0] = 0, query_start_loc[R] = T
 *   seq_lens               [R]       int32      KV length including this step's tokens
 *   block_table            [R, block_table_stride] int32 physical page ids
 * Query head h reads KV head h / (Hq / Hkv) (grouped-query attention).
 *
 * Ownership. The caller allocates and owns every buffer, device and host. The
 * library allocates no device memory, keeps no per-call state, and launches
 * only onto the stream it is given. out must not alias q, the caches or the
 * workspace. Device pointers must be 16-byte aligned.
 *
 * Errors. Every call returns a cb_status. Arguments and the host mirrors of
 * the metadata are validated before anything is launched; an invalid call
 * launches nothing. Page ids and slots live on the device and are bounds
 * checked there: an out-of-range one is skipped (it reads as zeros / is not
 * written) and its code is recorded in the workspace error word, which
 * cb_read_error_word returns. The library never aborts, traps or asserts on
 * the device.
 */
#ifndef CB_H
#define CB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum cb_status {
  CB_OK = 0,
  CB_ERR_INVALID_ARG = 1,   /* null pointer, bad size or dtype                         */
  CB_ERR_METADATA = 2,      /* host mirrors inconsistent (see cb_paged_attention)      */
  CB_ERR_UNSUPPORTED = 3,   /* shape outside the supported set                         */
  CB_ERR_WORKSPACE = 4,     /* workspace missing or smaller than cb_workspace_size()   */
  CB_ERR_CUDA = 5,          /* a CUDA runtime call failed; see cb_last_cuda_error()    */
  CB_ERR_DEVICE_CHECK = 6   /* returned by cb_read_error_word when the word is set     */
} cb_status;

typedef enum cb_dtype { CB_F32 = 0, CB_BF16 = 1 } cb_dtype;

/* Flags for cb_paged_attention. */
#define CB_FLAG_PORTABLE_ONLY 0x1u /* run every query row on the portable CUDA-core kernel */
/* For tests of the failure path only: one wait of each tensor-core attention
 * kernel (a consumer's first wait) is made to run out after a few polls. The
 * kernel then records CB_DEVERR_TIMEOUT, stops its other warps, waits for the
 * copies and products it has in flight, frees its tensor memory and returns;
 * the step's output is undefined. Call cb_workspace_init before the next step
 * on that workspace. */
#define CB_FLAG_TEST_WAIT_EXPIRY 0x2u

/* Error-word codes recorded on the device (bit set). */
#define CB_DEVERR_BLOCK_ID 0x1 /* a block_table entry outside [0, num_blocks) */
#define CB_DEVERR_SLOT 0x2     /* a slot_mapping entry >= num_blocks * block_size */
#define CB_DEVERR_TIMEOUT 0x4  /* a pipeline wait gave up (the kernel returned early) */

/* Static string for a status code; never NULL. */
const char* cb_status_string(int status);

/* Detail of the last failing call on the calling thread (static per thread); never NULL. */
const char* cb_last_error_message(void);

/* cudaError_t of the last failing CUDA call on the calling thread (0 if none). */
int cb_last_cuda_error(void);

/* ABI version of this header (incremented on any signature change). */
int cb_abi_version(void);
#define CB_ABI_VERSION 1

/*
 * cb_write_kv -- scatter the step's new K/V rows into their cache slots.
 *
 * Defined by the slot_mapping the scheduler builds ("Continuous Batching",
 * section "Extension: the vLLM v1 implementation"): for every token t with
 * slot_mapping[t] >= 0, k_cache viewed as [num_blocks * block_size, Hkv, D]
 * gets row slot_mapping[t] = k_new[t], and the same for V. Padding tokens may
 * point into the reserved pages 0-1 ("Continuous batching architecture",
 * section "Memory management") or use -1. A bit-exact copy.
 *
 * k_new, v_new: device [T, Hkv, D]; k_cache, v_cache: device caches (written);
 * slot_mapping: device int64 [T]. error_word: optional device int32 (NULL: no
 * record) that gets CB_DEVERR_SLOT or-ed in for a slot past the pool. Runs
 * asynchronously on `stream` (a cudaStream_t; NULL = legacy default stream).
 * Two tokens with the same non-negative slot race; which one wins is unspecified.
 */
cb_status cb_write_kv(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                      const int64_t* slot_mapping, int32_t num_tokens, int32_t num_blocks,
                      int32_t block_size, int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                      int32_t* error_word, void* stream);

/*
 * cb_copy_blocks -- batched copy of whole KV blocks: for every i < n, block
 * dst_ids[i] of (k_dst, v_dst) becomes block src_ids[i] of (k_src, v_src).
 *
 * The data movement of preemption by swapping and of CPU offloading: a request's
 * blocks are copied out to CPU memory and back into free pool blocks when it
 * resumes ("Continuous batching mechanics", d9bl.com, section "Running out of KV
 * cache memory"); the manager batches every offloaded request into one transfer
 * to a pinned CPU buffer ("Continuous batching architecture", Transformers docs,
 * section "Offloading"). The usual pattern: gather the blocks into a contiguous
 * device staging buffer with this call (dst_ids = 0 .. n-1), then one
 * cudaMemcpyAsync of the staging buffer to pinned host memory; the reverse on
 * resume. A bit-exact copy.
 *
 * k_src, v_src: device [src_num_blocks, block_size, Hkv, D]; k_dst, v_dst: device
 * [dst_num_blocks, block_size, Hkv, D] (written); src_ids, dst_ids: device int32
 * [n]. The source and destination may be the same buffers, provided no block is
 * both a source and a destination of the call; two pairs with the same
 * destination race (which one wins is unspecified). error_word: optional device
 * int32 (NULL: no record) that gets CB_DEVERR_BLOCK_ID or-ed in for a pair with an
 * id out of range (that pair is skipped). Runs asynchronously on `stream`.
 */
cb_status cb_copy_blocks(const void* k_src, const void* v_src, void* k_dst, void* v_dst,
                         int64_t src_num_blocks, int64_t dst_num_blocks, const int32_t* src_ids,
                         const int32_t* dst_ids, int32_t n, int32_t block_size,
                         int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                         int32_t* error_word, void* stream);

/*
 * cb_workspace_size -- bytes of device workspace cb_paged_attention needs for
 * a step with these sizes (an upper bound; it does not depend on the lengths).
 * The workspace holds the device error word and the split-KV partial results. One workspace serves every step of up to
 * num_requests requests with the same num_q_heads / num_kv_heads / head_dim:
 * its layout follows its size, not the step's request count, so steps of any
 * smaller size can share it (one stream at a time).
 */
size_t cb_workspace_size(int32_t num_requests, int32_t num_tokens, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim);

/*
 * cb_workspace_init -- zero the whole workspace (asynchronously on `stream`).
 * Call once after allocating a workspace, and again after a call recorded
 * CB_DEVERR_TIMEOUT; cb_read_error_word clears the error word.
 */
cb_status cb_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * cb_paged_attention -- one ragged mixed prefill/decode attention step.
 *
 * If k_new is not NULL the step first scatters k_new/v_new through
 * slot_mapping exactly as cb_write_kv does, then attends: the attended range
 * reaches this step's own tokens, which are read back from the cache.
 * slot_mapping must send each row to the slot of its own position (or < 0,
 * or to pages no request of the step reads, such as the reserved padding
 * pages), as a scheduler builds it: a step made of decode rows only (every
 * q_len <= 1) is run without a separate scatter launch -- the decode kernel
 * writes each row where it reads that position, so a slot pointing into a
 * position another request reads in the same step would race.
 * For every request r, row t = query_start_loc[r] + i (0 <= i < q_len) and
 * query head h, with g = h / (Hq / Hkv) and positions
 * p in [lo, context_len + i], lo = 0 or, with sliding_window W > 0,
 * max(0, context_len + i - W + 1):
 *     out[t, h] = sum_p softmax_p(scale * <q[t, h], K_p[g]>) * V_p[g]
 * accumulated in fp32 and rounded to the dtype of q.
 *
 * h_query_start_loc, h_seq_lens: host mirrors of the device metadata (the
 * same values). They are required: they are validated (query_start_loc[0] = 0,
 * non-decreasing, query_start_loc[R] = T; 0 <= q_len <= seq_len;
 * ceil(seq_len / block_size) <= block_table_stride) and used to plan the
 * launch. scale <= 0 selects 1/sqrt(head_dim). sliding_window <= 0 means full
 * causal attention.
 *
 * Supported: dtype CB_F32 or CB_BF16 (q, out, k_new, v_new and the caches in
 * that dtype); head_dim 64 or 128; Hq / Hkv in {1, 2, 4, 8, 16}; block_size a
 * power of two in [1, 256]. bf16 steps take the tensor-core paths where the
 * shape allows (decode rows: block_size a multiple of 16; prefill rows:
 * block_size a multiple of 8) and the portable CUDA-core kernel otherwise.
 *
 * workspace: device buffer of at least cb_workspace_size(...) bytes, zeroed
 * once by cb_workspace_init. Calls that share a workspace must be ordered on
 * one stream. Runs asynchronously on `stream`.
 */
cb_status cb_paged_attention(void* out, const void* q, void* k_cache, void* v_cache,
                             const void* k_new, const void* v_new, const int64_t* slot_mapping,
                             const int32_t* query_start_loc, const int32_t* seq_lens,
                             const int32_t* block_table, int32_t block_table_stride,
                             const int32_t* h_query_start_loc, const int32_t* h_seq_lens,
                             int32_t num_requests, int32_t num_tokens, int32_t num_blocks,
                             int32_t block_size, int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_dim, float scale, int32_t sliding_window, int32_t dtype,
                             uint32_t flags, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * cb_paged_attention_ring -- the same step for a sliding-window layer whose pages
 * are recycled in a ring: logical block b of request r lives in page
 * block_table[r * block_table_stride + b % ring_blocks] (the ring of a request has
 * ring_blocks entries; the rest of its row is unused).
 *
 * Sliding layers keep only a fixed window of recent tokens by reusing a small
 * number of pages, without a full per-request block table ("Continuous batching
 * architecture", Transformers docs, section "Memory management"). A position
 * older than the window may have been overwritten by a newer one mapping to the
 * same ring entry; it is never read. The caller builds slot_mapping with the same
 * mapping (slot = page_of(p) * block_size + p % block_size).
 *
 * Arguments, layouts, ownership and errors as cb_paged_attention, plus:
 * ring_blocks > 0 and <= block_table_stride, sliding_window > 0
 * (CB_ERR_INVALID_ARG otherwise), and for every request the positions from its
 * first query's window start max(0, context_len - sliding_window + 1) to
 * seq_len - 1 must span at most ring_blocks blocks, so that all of them are live
 * at once (CB_ERR_METADATA otherwise).
 */
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
                                  size_t workspace_bytes, void* stream);

/*
 * CUDA graphs of the step, one per padded shape.
 *
 * Every step costs CPU time to assemble and launch; recording the GPU work once
 * and replaying it for batches of the same padded shape removes that cost. The
 * query length is padded to a multiple of q_padding_interval_size and the KV
 * length to a multiple of kv_padding_interval_size; recorded graphs are kept in a
 * cache and a batch whose padded shape matches one is replayed without CPU
 * scheduling, while a new shape triggers a capture ("Continuous batching
 * architecture", Transformers docs, section "CUDA graphs").
 *
 * cb_graph_cache_create -- an empty cache; q_interval > 0 (the query-length
 * padding interval), kv_interval >= 0 (the KV-length bucket; 0: one bucket, as
 * the launches here do not depend on the KV length). Owned by the caller, freed
 * with cb_graph_cache_destroy (which destroys its graphs). Not tied to a device
 * until the first call; all calls on one cache must use the same device.
 */
typedef struct cb_graph_cache cb_graph_cache;
cb_status cb_graph_cache_create(int32_t q_interval, int32_t kv_interval, cb_graph_cache** cache);
void cb_graph_cache_destroy(cb_graph_cache* cache);
/* Number of graphs held, captures made and replays served; any pointer may be NULL. */
cb_status cb_graph_cache_stats(cb_graph_cache* cache, int64_t* graphs, int64_t* captures,
                               int64_t* replays);

/*
 * cb_paged_attention_graphed -- cb_paged_attention, captured into a CUDA graph the
 * first time its key is seen and replayed afterwards. The key is every buffer
 * pointer, every size, num_requests and num_tokens (the padded counts), the
 * KV-length bucket and whether the batch has decode rows and prefill rows (so a
 * graph holds only the launches its batches need); the metadata values are read on the device at
 * replay (the decode kernel sums its work and the prefill kernel finds its tiles
 * there), so one graph serves every batch of its shape. Arguments as
 * cb_paged_attention, with the padded shape:
 *   num_requests and num_tokens multiples of q_interval (CB_ERR_INVALID_ARG);
 *   requests past the real ones have q_len 0 and seq_len 0; tokens past
 *   query_start_loc[R] are padding (slot_mapping -1, their out rows untouched);
 *   query_start_loc[R] <= num_tokens.
 * The caller keeps the buffers alive and in place while the cache holds graphs
 * that name them, writes each step's inputs into them before the call, and must
 * not pass the legacy default stream. Supported: bf16 with shapes that the split-KV
 * decode and the tile prefill kernels both cover (CB_ERR_UNSUPPORTED otherwise).
 * Per-kernel timing (cb_kernel_timing) does not see replayed kernels; the launch
 * counts do. Thread-safe per cache (one mutex).
 */
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
                                     size_t workspace_bytes, void* stream);

/*
 * cb_read_error_word -- synchronise `stream`, copy the workspace error word
 * to *h_error, clear it, and return CB_ERR_DEVICE_CHECK if it was non-zero.
 */
cb_status cb_read_error_word(void* workspace, int32_t* h_error, void* stream);

/*
 * cb_paged_attention_no_alloc -- cb_paged_attention for callers that may not
 * allocate device memory when they call the library: for instance a plugin
 * inside a host program that owns the device memory pool and forbids
 * allocations on its inference path, or a latency-critical caller that cannot
 * pay the implicit device synchronisation of cudaMalloc/cudaFree. The pages
 * define nothing like it: it is a deployment convenience of this library.
 *
 * Arguments and results are those of cb_paged_attention without the workspace
 * pair. The scratch the step needs lives instead in one fixed device array of
 * CB_NO_ALLOC_SCRATCH_BYTES compiled into the library; every GPU that loads the
 * library holds it until the process exits. The call allocates and frees
 * nothing. A step whose plan needs more scratch than the array is rejected
 * with CB_ERR_WORKSPACE and nothing is launched (at 8 MiB the array covers,
 * for example, 64 decode requests with 32 query heads of size 128, or 16 with
 * 64 heads).
 *
 * The first call on a device looks up the array's device address with that
 * device current and caches it; make that first call before any stream
 * capture. Every call shares the one array and finds it holding the previous
 * call's contents; the call clears the part that must start at zero (the error
 * word) on `stream` before its kernels. Calls whose
 * work overlaps on the GPU (other streams, other host threads) race on the
 * array: order them on one stream. The device error word lives in the array:
 * read it with cb_no_alloc_read_error_word (below) after a call and before the
 * next one, which clears it.
 */
#define CB_NO_ALLOC_SCRATCH_BYTES (8u << 20)
cb_status cb_paged_attention_no_alloc(void* out, const void* q, void* k_cache, void* v_cache,
                                      const void* k_new, const void* v_new,
                                      const int64_t* slot_mapping,
                                      const int32_t* query_start_loc, const int32_t* seq_lens,
                                      const int32_t* block_table, int32_t block_table_stride,
                                      const int32_t* h_query_start_loc, const int32_t* h_seq_lens,
                                      int32_t num_requests, int32_t num_tokens, int32_t num_blocks,
                                      int32_t block_size, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, float scale,
                                      int32_t sliding_window, int32_t dtype, uint32_t flags,
                                      void* stream);

/*
 * cb_no_alloc_read_error_word -- cb_read_error_word for the error word of
 * cb_paged_attention_no_alloc (which lives in the library's fixed scratch
 * array, not in a caller's workspace): synchronise `stream`, copy the word of
 * the current device to *h_error, clear it, and return CB_ERR_DEVICE_CHECK if
 * it was non-zero. Allocates nothing. The next cb_paged_attention_no_alloc
 * call clears the word as well, so read it in between.
 */
cb_status cb_no_alloc_read_error_word(int32_t* h_error, void* stream);

/* ---- diagnostics (no effect on results) -------------------------------- */

/* Number of kernels the library has launched in this process: of kernel id
 * `kernel` (0 .. cb_num_kernels()-1), or of all kernels when kernel < 0. */
long long cb_launch_count(int kernel);

/* Number of kernel ids, and the static name of one ("" when out of range). */
int cb_num_kernels(void);
const char* cb_kernel_name(int kernel);

/* When enabled (per calling thread), every kernel launch is bracketed by a
 * pair of CUDA events on its stream, so per-kernel device time can be read. */
cb_status cb_kernel_timing(int enable);

/* Synchronise the recorded events and return, per kernel id (n entries), the
 * total milliseconds and the launch count since the previous collect. */
cb_status cb_kernel_timing_collect(double* total_ms, long long* launches, int n);

#ifdef __cplusplus
}
#endif

#endif /* CB_H */
