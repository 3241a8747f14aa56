// realise.cu -- turning a balanced layout into sharded weights
// ("Affinity-Aware Sharding for Delayed Tensor Parallelism", §3 "The layout
// as a free variable"): KV groups and neurons are put in order of device
// (stable within a device), the query/key/value rows follow their group
// (each group with its query heads), the output-projection columns follow the
// query heads, gate/up rows and down columns follow the neurons; device l's
// shard is then the l-th contiguous slice of every permuted matrix.
#include "affinity.h"
#include "internal.h"

#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

namespace aff {
namespace {

// out[r][j] = in[r][order[j]] for blocks of `B` bytes, rows of n_blocks * B
// bytes.  Each thread moves one W-byte word; W divides B and both pointers.
template <typename Word>
__global__ void gather_blocks_kernel(const Word* __restrict__ in, Word* __restrict__ out, int64_t rows,
                                     int64_t n_blocks, int64_t words_per_block, const int32_t* __restrict__ order) {
  const int64_t per_row = n_blocks * words_per_block;
  const int64_t total = rows * per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / per_row;
    const int64_t rem = i - r * per_row;
    const int64_t j = rem / words_per_block;
    const int64_t w = rem - j * words_per_block;
    out[i] = in[r * per_row + (int64_t)__ldg(order + j) * words_per_block + w];
  }
}

template <typename Word>
aff_status launch_gather(const void* in, void* out, int64_t rows, int64_t n_blocks, int64_t block_bytes,
                         const int32_t* order, cudaStream_t s, int sms) {
  const int64_t wpb = block_bytes / (int64_t)sizeof(Word);
  const int64_t total = rows * n_blocks * wpb;
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)sms * 8;
  gather_blocks_kernel<Word><<<(unsigned)(want < cap ? want : cap), threads, 0, s>>>(
      static_cast<const Word*>(in), static_cast<Word*>(out), rows, n_blocks, wpb, order);
  AFF_CUDA(cudaGetLastError());
  return AFF_OK;
}

}  // namespace
}  // namespace aff

using namespace aff;

extern "C" {

aff_status affinity_layout_orders(const int32_t* h, const int32_t* nu, int32_t G, int64_t H, int64_t I, int32_t L,
                                  int32_t* group_order, int32_t* head_order, int32_t* neuron_order) {
  if (!h || !nu || !group_order || !head_order || !neuron_order) return AFF_ERR_INVALID_ARG;
  if (G < 1 || H < G || H % G || I < 1 || L < 1 || G % L || I % L) return AFF_ERR_INVALID_ARG;
  std::vector<int64_t> gc(L, 0), nc(L, 0);
  for (int g = 0; g < G; ++g) {
    if (h[g] < 0 || h[g] >= L) return AFF_ERR_INVALID_ARG;
    gc[h[g]]++;
  }
  for (int64_t k = 0; k < I; ++k) {
    if (nu[k] < 0 || nu[k] >= L) return AFF_ERR_INVALID_ARG;
    nc[nu[k]]++;
  }
  for (int l = 0; l < L; ++l)
    if (gc[l] != G / L || nc[l] != I / L) return AFF_ERR_INVALID_ARG;
  // stable counting sort by device
  int64_t pos = 0;
  for (int l = 0; l < L; ++l)
    for (int g = 0; g < G; ++g)
      if (h[g] == l) group_order[pos++] = g;
  const int64_t hpg = H / G;
  for (int i = 0; i < G; ++i)
    for (int64_t j = 0; j < hpg; ++j) head_order[i * hpg + j] = (int32_t)(group_order[i] * hpg + j);
  pos = 0;
  for (int l = 0; l < L; ++l)
    for (int64_t k = 0; k < I; ++k)
      if (nu[k] == l) neuron_order[pos++] = (int32_t)k;
  return AFF_OK;
}

aff_status affinity_gather_blocks(const void* in, void* out, int64_t rows, int64_t n_blocks, int64_t block_bytes,
                                  const int32_t* order, void* workspace, size_t workspace_bytes,
                                  aff_stream_t stream) {
  if (!in || !out || !order || rows < 1 || n_blocks < 1 || block_bytes < 1) return AFF_ERR_INVALID_ARG;
  if (n_blocks > INT32_MAX) return AFF_ERR_UNSUPPORTED_SHAPE;
  const char* ib = static_cast<const char*>(in);
  const char* ob = static_cast<const char*>(out);
  const int64_t bytes = rows * n_blocks * block_bytes;
  if (ib < ob + bytes && ob < ib + bytes) return AFF_ERR_INVALID_ARG;  // overlapping buffers
  // the order must be a permutation of 0..n_blocks-1: then every read is in bounds
  std::vector<uint8_t> seen((size_t)n_blocks, 0);
  for (int64_t j = 0; j < n_blocks; ++j) {
    if (order[j] < 0 || order[j] >= n_blocks || seen[order[j]]) return AFF_ERR_INVALID_ARG;
    seen[order[j]] = 1;
  }
  if (!workspace || workspace_bytes < (size_t)n_blocks * sizeof(int32_t) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return AFF_ERR_WORKSPACE;
  int sms = 0;
  aff_status st = check_device(&sms);
  if (st != AFF_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* d_order = static_cast<int32_t*>(workspace);
  AFF_CUDA(cudaMemcpyAsync(d_order, order, (size_t)n_blocks * sizeof(int32_t), cudaMemcpyHostToDevice, s));
  const uintptr_t a = reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out);
  if (block_bytes % 16 == 0 && (a & 15u) == 0)
    return launch_gather<uint4>(in, out, rows, n_blocks, block_bytes, d_order, s, sms);
  if (block_bytes % 8 == 0 && (a & 7u) == 0)
    return launch_gather<uint2>(in, out, rows, n_blocks, block_bytes, d_order, s, sms);
  if (block_bytes % 4 == 0 && (a & 3u) == 0)
    return launch_gather<uint32_t>(in, out, rows, n_blocks, block_bytes, d_order, s, sms);
  if (block_bytes % 2 == 0 && (a & 1u) == 0)
    return launch_gather<uint16_t>(in, out, rows, n_blocks, block_bytes, d_order, s, sms);
  return launch_gather<uint8_t>(in, out, rows, n_blocks, block_bytes, d_order, s, sms);
}

}  // extern "C"
