// Decode split-KV kernel: arguments shared by the host planner and the kernels.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.h"

namespace cb {

constexpr int kDecodeMaxStages = 8;
constexpr int kDecodeMaxHeads = 8;          // KV heads per CTA (one consumer warp each)
constexpr int kDecodeSmemLimit = 232448;    // 227 KiB dynamic shared memory per CTA
constexpr int kDecodeTableCtas = 256;       // CTAs whose start is passed in the arguments
constexpr int kDecodeMinBlocksPerCta = 4;   // key blocks per CTA at least (small steps)
constexpr int CB_DEVERR_BLOCK_ID_CODE = 0x1;
constexpr int CB_DEVERR_SLOT_CODE = 0x2;
constexpr int CB_DEVERR_TIMEOUT_CODE = 0x4;

// Where CTA b's range of key blocks starts, placed by the host from its mirrors of
// the metadata, so that the CTA's first copies wait on one load (its page ids).
struct DecodeCtaStart {
  int r;    // first request (-1: none)
  int u_r;  // global index of that request's first key block
  int kb0;  // first key block (within the request) of the CTA's first segment
  int kb1;  // one past its last key block
  int t;    // packed query row of the request
  int seq;  // its seq_len
};

struct DecodeArgs {
  StepArgs a;
  long long total_units;  // key blocks of all decode requests
  int num_ctas;           // C
  int heads_per_cta;      // HB
  int stages;
  int stage_bytes;        // K + V of one 16-key block for HB heads
  int q_slot_bytes;       // HB * G * D * 2
  int metadata_ready;     // the step's previous kernel is libcb's scatter
  int units_on_device;    // total_units is summed by the kernel from the device metadata
                          // (graph replays: nothing in the arguments depends on the batch)
  float* part_o;          // [slots][Hq][D] unnormalised partial outputs
  float2* part_ml;        // [slots][Hq] (running max in log2 units, sum)
  // Steps of decode rows only: the CTA that reads a request's last key block writes
  // the request's new K/V row (its heads) into the row's slot and into its staged
  // copy of that block, so the step needs no separate scatter launch. The row's slot
  // must be that of the request's last position (or < 0: not written), as a
  // scheduler-built slot_mapping has it.
  int fuse_scatter;
  const void* k_new;      // [T, Hkv, D]
  const void* v_new;
  const int64_t* slot_mapping;
  int has_table;          // cta_first is filled (num_ctas <= kDecodeTableCtas)
  DecodeCtaStart cta_first[kDecodeTableCtas];
};

struct DecodePlan {
  size_t smem_bytes;
};

// A request whose key blocks span several decode CTAs (b_first .. b_first + nseg - 1):
// its partials sit in slots r + b_first .. r + b_first + nseg - 1.
struct CombineEntry {
  int r;
  int t;        // its packed query row
  int b_first;
  int nseg;
};

constexpr int kCombineListMax = 256;    // split requests the host lists in the arguments
constexpr int kCombineMaxThreads = 512;  // per CTA: four outputs of its KV heads each, x parts
constexpr int kCombineSegmentsInFlight = 12;  // partials a combine thread loads at once

struct CombineArgs {
  StepArgs a;
  int num_ctas;           // C of the decode launch (its partition: CTA b takes [b U/C, (b+1) U/C))
  const float* part_o;    // the decode launch's partials
  const float2* part_ml;
  int kv_per_cta;         // KV heads merged by one CTA (divides num_kv_heads; x G x D / 4 <= 512)
  int parts;              // threads per output (each merges a share of the segments; >= 1)
  int n_entries;  // >= 0: entries[0 .. n_entries) are the split requests; -1: the
                  // kernel finds them from the device metadata (one CTA per request)
  CombineEntry entries[kCombineListMax];
};

size_t decode_smem_bytes(int stages, int stage_bytes, int q_slot_bytes);
cudaError_t launch_decode(DecodeArgs p, const DecodePlan& plan, cudaStream_t stream);
// The merge of the split requests' partials, on the stream right after launch_decode.
cudaError_t launch_decode_combine(const CombineArgs& c, cudaStream_t stream);
// Kernel attributes the launch needs, set without launching (before a stream capture).
cudaError_t prepare_decode(const DecodeArgs& p);

}  // namespace cb
