// Launch accounting and optional per-kernel CUDA-event timing (diagnostics).
//
// Every kernel launch of the library goes through launch_pdl, which bumps a
// process-wide counter per kernel and, when timing is enabled on the calling
// thread, brackets the launch with a pair of CUDA events on its stream.
#include <cuda_runtime.h>

#include <atomic>
#include <vector>

#include "cb.h"
#include "launch.h"

namespace cb {
namespace {

std::atomic<long long> g_launches[kNumKernels];

struct Pending {
  int kernel;
  cudaEvent_t start, stop;
};

thread_local bool t_timing = false;
thread_local std::vector<Pending> t_pending;
thread_local std::vector<cudaEvent_t> t_free_events;
thread_local double t_ms[kNumKernels];
thread_local long long t_count[kNumKernels];
thread_local cudaEvent_t t_open_start = nullptr;

cudaEvent_t take_event() {
  if (!t_free_events.empty()) {
    cudaEvent_t e = t_free_events.back();
    t_free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

const char* const kNames[kNumKernels] = {"write_kv", "portable_attention", "decode_split",
                                         "prefill_tc", "copy_blocks", "decode_combine"};

}  // namespace

void note_launch_begin(KernelId id, cudaStream_t stream) {
  g_launches[id].fetch_add(1, std::memory_order_relaxed);
  if (!t_timing) return;
  t_open_start = take_event();
  if (t_open_start) cudaEventRecord(t_open_start, stream);
}

void note_launch_end(KernelId id, cudaStream_t stream) {
  if (!t_timing || !t_open_start) return;
  cudaEvent_t stop = take_event();
  if (!stop) return;
  cudaEventRecord(stop, stream);
  t_pending.push_back({(int)id, t_open_start, stop});
  t_open_start = nullptr;
}

void note_replayed_launches(const long long* per_kernel) {
  for (int k = 0; k < kNumKernels; ++k)
    g_launches[k].fetch_add(per_kernel[k], std::memory_order_relaxed);
}

void launch_counts(long long* per_kernel) {
  for (int k = 0; k < kNumKernels; ++k) per_kernel[k] = g_launches[k].load();
}

bool set_kernel_timing(bool enable) {
  const bool was = t_timing;
  t_timing = enable;
  return was;
}

}  // namespace cb

extern "C" {

long long cb_launch_count(int kernel) {
  if (kernel < 0) {
    long long s = 0;
    for (int k = 0; k < cb::kNumKernels; ++k) s += cb::g_launches[k].load();
    return s;
  }
  if (kernel >= cb::kNumKernels) return 0;
  return cb::g_launches[kernel].load();
}

const char* cb_kernel_name(int kernel) {
  if (kernel < 0 || kernel >= cb::kNumKernels) return "";
  return cb::kNames[kernel];
}

int cb_num_kernels(void) { return cb::kNumKernels; }

cb_status cb_kernel_timing(int enable) {
  cb::t_timing = enable != 0;
  return CB_OK;
}

cb_status cb_kernel_timing_collect(double* total_ms, long long* launches, int n) {
  for (auto& p : cb::t_pending) {
    if (cudaEventSynchronize(p.stop) != cudaSuccess) return CB_ERR_CUDA;
    float ms = 0.f;
    cudaEventElapsedTime(&ms, p.start, p.stop);
    cb::t_ms[p.kernel] += ms;
    cb::t_count[p.kernel] += 1;
    cb::t_free_events.push_back(p.start);
    cb::t_free_events.push_back(p.stop);
  }
  cb::t_pending.clear();
  for (int k = 0; k < n && k < cb::kNumKernels; ++k) {
    if (total_ms) total_ms[k] = cb::t_ms[k];
    if (launches) launches[k] = cb::t_count[k];
    cb::t_ms[k] = 0.0;
    cb::t_count[k] = 0;
  }
  return CB_OK;
}

}  // extern "C"
