// Prefill / chunked-prefill tile kernel: arguments shared by the planner and the kernel.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.h"

namespace cb {

constexpr int kPrefillMaxEntries = 128;  // prefill requests per launch (more: several launches)
constexpr int kPrefillSmemLimit = 232448;

// One prefill request of the step: its index and number of query tiles.
struct PrefillEntry {
  int r;
  int n_qtiles;
};

struct PrefillArgs {
  StepArgs a;
  int tile_tokens;   // query tokens per 128-row tile (128 / G)
  int box_keys;      // keys per page box: min(block_size, 128)
  int n_entries;
  int total_ctas;    // sum of n_qtiles * Hkv
  PrefillEntry entries[kPrefillMaxEntries];  // heaviest first
};

size_t prefill_smem_bytes(int head_dim);
// Launch the tile kernel over the prefill requests listed in `p` (already sorted).
cudaError_t launch_prefill(const PrefillArgs& p, cudaStream_t stream);

}  // namespace cb
