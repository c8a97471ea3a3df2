// Prefill / chunked-prefill tile kernel: arguments shared by the planner and the kernel.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.h"

namespace cb {

constexpr int kPrefillMaxEntries = 128;  // prefill requests per launch (more: several launches)
constexpr int kPrefillSmemLimit = 232448;

// One prefill request of the step: its index, number of query tiles, and its
// query_start_loc / q_len / seq_len as the planner read them from the host
// copies (so that a CTA needs no dependent metadata loads before its work).
struct PrefillEntry {
  int r;
  int n_qtiles;
  int q_start;
  int q_len;
  int seq_len;
};

struct PrefillArgs {
  StepArgs a;
  int tile_tokens;   // query tokens per 128-row tile (128 / G)
  int box_keys;      // keys per page box: min(block_size, 128)
  int n_entries;
  int metadata_ready;  // a libcb kernel precedes this one in the step: q and the metadata are visible
  int total_ctas;    // sum over entries of prefill_ctas(n_qtiles, Hkv)
  PrefillEntry entries[kPrefillMaxEntries];  // heaviest first
};

size_t prefill_smem_bytes(int head_dim);
// CTAs the tile kernel runs for one request of n_qtiles query tiles.
int prefill_ctas(int n_qtiles, int num_kv_heads);
// Launch the tile kernel over the prefill requests listed in `p` (already sorted).
cudaError_t launch_prefill(const PrefillArgs& p, cudaStream_t stream);

}  // namespace cb
