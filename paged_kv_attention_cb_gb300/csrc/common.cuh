// Device helpers shared by the libcb kernels (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define CB_DEV __device__ __forceinline__

namespace cb {

// Programmatic dependent launch: every kernel is launched so that it may start
// while the previous kernel on the stream drains; it must wait for that kernel
// (and see its writes) before touching global inputs.
CB_DEV void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
CB_DEV void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

CB_DEV void record_error(int32_t* word, int code) {
  if (word != nullptr) atomicOr(word, code);
}

template <typename T> struct Elt;
template <> struct Elt<float> {
  static CB_DEV float to_f(float x) { return x; }
  static CB_DEV float from_f(float x) { return x; }
};
template <> struct Elt<__nv_bfloat16> {
  static CB_DEV float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static CB_DEV __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// Block-table entry of logical block `b`: entry b of the request's row, or, for a
// sliding layer whose pages are recycled in a ring of `ring` pages ("Continuous
// batching architecture", Transformers docs, section "Memory management": sliding
// layers keep only a window of recent tokens by reusing a small number of pages),
// entry b % ring.
CB_DEV int bt_entry(int b, int ring) { return ring > 0 ? b % ring : b; }

// log2(e): the kernels keep scores in the base-2 domain (exp2 on the SFU).
constexpr float kLog2e = 1.4426950408889634f;

}  // namespace cb
