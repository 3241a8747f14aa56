// launch.cuh -- programmatic dependent launch for the kernels of one call.
//
// The kernels of an affinity_up / affinity_down call form short chains on one
// or two streams, and several of them run for only a few microseconds, so the
// gap between one kernel's end and the next one's start is a visible share of
// a call.  They are launched with programmatic stream serialisation: the next
// kernel in a stream is scheduled as the previous one's blocks finish (or, for
// a kernel that calls pdl_launch_dependents, as soon as all of its blocks have
// started), and its first statement, pdl_wait(), blocks until the previous
// kernel has completed and its writes are visible.  Nothing is read or written
// before that wait, so the results are those of plain stream order.
// AFFINITY_PDL=0 launches them plainly.
//
// Measured on the Qwen3-shaped layer (steps, ms, against plain launches): ADD
// 0.1889 -> 0.1811, down 1.0783 -> 1.0571, LOO 2.6903 -> 2.6821, FO 2.0675 ->
// 2.0614 (a box held below its top clock).  Signalling at the start of every
// kernel instead made ADD and LOO slower: the next kernel's blocks then sat on
// SMs that a kernel on the other stream was waiting for.
#pragma once

#include <cuda_runtime.h>

#include <cstdlib>
#include <utility>

namespace aff {

#ifdef __CUDACC__
// Wait for the previous kernel in the stream (a no-op when launched plainly).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel in the stream to be scheduled.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// The first statement of every kernel launched by launch_pdl.
__device__ __forceinline__ void pdl_enter() { pdl_wait(); }
#endif

inline bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("AFFINITY_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace aff
