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
  // The step's new K/V rows (nullptr: none, or already in the cache). With them the
  // kernel reads a request's own new positions from k_new / v_new instead of the
  // cache -- each position whose slot_mapping entry is its own slot, which is the
  // value the cache will hold -- and its CTAs copy the rows of every listed request
  // into their slots (claimed in parts once their units are done), so the step needs no
  // scatter launch and nothing in it reads a position written in it.
  const void* k_new;
  const void* v_new;
  const int64_t* slot_mapping;
  // Launched right after the decode kernel of the step (programmatic dependent launch),
  // while the decode CTAs stream: the kernel needs nothing they write, so it does not
  // wait for them; the last of its CTAs to finish waits for the decode grid, so that the
  // completion of this grid implies the decode grid's (the combine launch that follows
  // reads the decode partials). exit_counter: an int in the workspace header, zero
  // between steps (the last CTA also resets unit_counter through it).
  int concurrent;
  int* exit_counter;
  int device_work;     // entries unused: each CTA finds its work in the device metadata (graph
                       // replays: nothing in the arguments depends on the batch); total_ctas is
                       // then an upper bound and the CTAs past the step's work exit at once
  int total_ctas;    // units: sum over entries of prefill_ctas(n_qtiles, Hkv) (an upper bound
                     // with device_work)
  int total_units;   // units of the list (CTAs claim them through unit_counter)
  int grid;          // CTAs launched: min(units, SMs); with device_work one per unit (bound)
  int* unit_counter; // next unit of the list to claim (workspace header, zero between steps)
  int* scatter_counter;  // next part of the new-row copy to claim (likewise)
  PrefillEntry entries[kPrefillMaxEntries];  // heaviest first
};

size_t prefill_smem_bytes(int head_dim);
// Most prefill CTAs a step of up to `num_tokens` query tokens in `num_requests`
// requests can need (the grid of a launch whose work is found on the device).
int prefill_ctas_bound(int num_tokens, int num_requests, int tile_tokens, int num_kv_heads);
// CTAs the tile kernel runs for one request of n_qtiles query tiles.
int prefill_ctas(int n_qtiles, int num_kv_heads);
// Launch the tile kernel over the prefill requests listed in `p` (already sorted).
cudaError_t launch_prefill(const PrefillArgs& p, cudaStream_t stream);
// Kernel attributes the launch needs, set without launching (before a stream capture).
cudaError_t prepare_prefill(int head_dim);

}  // namespace cb
