// noalloc.cu -- affinity_up_static: affinity_up for callers that cannot
// allocate device memory, with its scratch space compiled into the library.
#include "affinity.h"

#include <cuda_runtime.h>

#include <mutex>
#include <vector>

namespace {

// Scratch used in place of a caller-provided workspace.  Every GPU on which
// this module is loaded holds these bytes until the process exits.  The
// module is compiled on its own, so under CUDA's lazy module loading (the
// default) it is loaded on a device, and the 64 MiB reserved there, at the
// first symbol lookup below: the first affinity_up_static or
// affinity_static_device_status call on that device.
constexpr size_t kStaticScratchBytes = 64ull << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device.  In host code the
// array's name only stands in for the symbol; a kernel must be given this
// address instead.  Looked up once per device, with that device current.
aff_status scratch_on_current_device(void** out) {
  static std::mutex mu;
  static std::vector<void*> addr;  // per device ordinal; nullptr until looked up
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return AFF_ERR_ARCH;
  }
  std::lock_guard<std::mutex> lk(mu);
  if ((int)addr.size() <= dev) addr.resize(dev + 1, nullptr);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return AFF_ERR_CUDA;
    }
    addr[dev] = p;
  }
  *out = addr[dev];
  return AFF_OK;
}

}  // namespace

extern "C" aff_status affinity_up_static(const void* a, const void* x, const void* Wo, const void* gamma,
                                         const void* Wg, const void* Wu, const void* Wd, const aff_dims* dims,
                                         int32_t mode, float* S_out, float* S_head_out, aff_stream_t stream) {
  size_t need = 0;
  aff_status st = affinity_workspace_size(dims, mode, 0, &need);
  if (st != AFF_OK) return st;
  if (need > kStaticScratchBytes) return AFF_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((st = scratch_on_current_device(&scratch)) != AFF_OK) return st;
  // Every buffer the pass reads is written earlier in the same call (the
  // status word is cleared at its start), so leftovers of a previous call
  // in the shared array never reach the result.
  return affinity_up(a, x, Wo, gamma, Wg, Wu, Wd, dims, mode, S_out, S_head_out, scratch, kStaticScratchBytes,
                     stream);
}

// The status word of the static scratch sits where a workspace keeps it, at
// offset 0, so reading it is affinity_device_status on the array's address.
extern "C" aff_status affinity_static_device_status(aff_stream_t stream) {
  void* scratch = nullptr;
  const aff_status st = scratch_on_current_device(&scratch);
  if (st != AFF_OK) return st;
  return affinity_device_status(scratch, stream);
}
