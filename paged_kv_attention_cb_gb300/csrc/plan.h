// Work partition of one step (host side): which kernel serves which query rows,
// and how the decode rows' KV is split across CTAs.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "decode.h"
#include "prefill.h"
#include "launch.h"

namespace cb {

constexpr size_t kWorkspaceHeaderBytes = 256;  // error word, prefill exit counter, reserved
constexpr size_t kExitCounterOffset = 64;      // int: prefill CTAs finished (zero between steps)
constexpr size_t kUnitCounterOffset = 128;     // int: prefill units claimed (zero between steps)
constexpr size_t kScatterCounterOffset = 192;  // int: prefill row-copy parts claimed (likewise)
constexpr int kMaxDecodeCtas = 2048;           // upper bound on decode CTAs (workspace sizing)
constexpr int kMaxPrefillLaunches = 8;         // x kPrefillMaxEntries prefill requests per step

size_t workspace_bytes(int32_t num_requests, int32_t num_tokens, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim);

// The step's new K/V rows: cb_paged_attention's k_new / v_new / slot_mapping.
struct ScatterInputs {
  const void* k_new;
  const void* v_new;
  const int64_t* slot_mapping;
};

struct Plan {
  int portable_mode;   // -1: none, 0: all rows, 1: decode rows, 2: prefill rows
  bool fast_decode;    // decode rows on the split-KV tensor-core kernel
  bool fast_prefill;   // prefill rows on the tcgen05 tile kernel
  bool fused_scatter;  // the attention kernels write the new K/V rows (no scatter launch)
  bool concurrent;     // decode and prefill grids run side by side (decode, prefill, combine)
  void* workspace;
  size_t workspace_bytes;
  DecodeArgs decode;
  DecodePlan decode_plan;
  bool has_combine;     // a combine launch follows the decode launch
  CombineArgs combine;
  int n_prefill_launches;
  PrefillArgs prefill[kMaxPrefillLaunches];
};

// scatter: the step's new rows (nullptr: none). Unless the plan fuses them into the
// decode kernel (fused_scatter), the caller launches the scatter before run_plan.
void plan_step(Plan& plan, const StepArgs& a, const int32_t* h_qsl, const int32_t* h_seq_lens,
               uint32_t flags, const ScatterInputs* scatter, void* workspace,
               size_t workspace_bytes);

cudaError_t run_plan(const Plan& plan, const StepArgs& a, cudaStream_t stream);

// A plan whose launches depend only on the step's padded shape (a.num_requests,
// a.num_tokens) and static sizes, for capture in a CUDA graph that is replayed for
// every batch of that shape: the decode kernel sums its work on the device and the
// prefill kernel finds its tiles in the device metadata. False when the shape
// needs a kernel this mode does not cover (fp32, or a decode/prefill case only the
// portable kernel runs). with_decode / with_prefill: whether the graph has the
// decode / prefill launch (the batches it serves have rows of that kind).
bool plan_graph_step(Plan& plan, const StepArgs& a, bool with_decode, bool with_prefill,
                     void* workspace, size_t workspace_bytes);
// Set the kernel attributes of the plan's launches (before a capture).
cudaError_t prepare_plan(const Plan& plan, const StepArgs& a);

// Bytes at the start of the workspace that the planned launch reads or writes
// (the rest of a cb_workspace_size() buffer is headroom for larger plans), and
// the leading part of it that must be zero before a call (the error word).
// The workspace's layout depends on its size only, never on the step's request
// count, so that steps of any size can share one workspace.
size_t workspace_extent(const Plan& plan, const StepArgs& a);
size_t workspace_zeroed_prefix(const StepArgs& a, size_t workspace_bytes);

}  // namespace cb
