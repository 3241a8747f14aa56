// internal.h -- helpers shared by the translation units behind the C ABI
// (not part of include/affinity.h).
#pragma once

#include "affinity.h"

#include <cuda_runtime.h>

namespace aff {

// Records "<where>: <CUDA error name> (<text>)" for affinity_last_cuda_error()
// on this thread and returns AFF_ERR_CUDA.
aff_status cuda_fail(cudaError_t e, const char* where);

// AFF_OK with the SM count when the current device is an sm_103 part;
// AFF_ERR_ARCH otherwise (also when there is no device).
aff_status check_device(int* sm_count);

}  // namespace aff

#define AFF_CUDA(call)                                        \
  do {                                                        \
    cudaError_t e_ = (call);                                  \
    if (e_ != cudaSuccess) return ::aff::cuda_fail(e_, #call); \
  } while (0)
