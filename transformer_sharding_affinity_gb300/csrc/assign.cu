// assign.cu -- the neuron step of the layout search on the GPU and the
// alternating optimiser around it ("Affinity-Aware Sharding for Delayed
// Tensor Parallelism", §3 "Optimiser").
//
// Given the KV-group maps h_i and h_{i+1}, putting neuron k of layer i on
// device l gains M[k, l] = sum_{g: h_i(g)=l} Shat_up_i[g, k]
//                        + sum_{g: h_{i+1}(g)=l} Shat_down_i[k, g],
// and the best balanced neuron map (I/L neurons per device) maximises
// sum_k M[k, nu(k)].  The solver follows the paper's outline -- dual ascent
// on the L device offsets, a fix-up to meet the capacities exactly, then
// local exchanges -- but the exchanges are not limited to pairs: any cycle
// of devices that moves one neuron out of each device on it is applied while
// it gains, so the result is the exact optimum of the transportation problem
// (a balanced map is optimal exactly when no such cycle gains).
#include "affinity.h"
#include "internal.h"

#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>
#include <cstring>
#include <vector>

namespace aff {
namespace {

constexpr int kAssignThreads = 1024;
constexpr int kWarps = kAssignThreads / 32;
constexpr int kMaxL = 8;
constexpr int kMaxG = 16;
constexpr int64_t kMaxNeurons = 49152;  // the map lives in shared memory (4 B per neuron)

// ------------------------------------------------------------------ gain M
struct GainParams {
  const double* Su;  // [G][I]
  const double* Sd;  // [I][G] or null
  double* M;         // [I][L]
  int64_t I;
  int G, L;
  int8_t h[kMaxG], hn[kMaxG];
};

__global__ void neuron_gain_kernel(GainParams p) {
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= p.I) return;
  double m[kMaxL];
#pragma unroll
  for (int l = 0; l < kMaxL; ++l) m[l] = 0.0;
  // same order of additions as the definition: groups ascending, up then down
  for (int g = 0; g < p.G; ++g) {
    const double v = p.Su[(size_t)g * p.I + k];
#pragma unroll
    for (int l = 0; l < kMaxL; ++l)
      if (l == p.h[g]) m[l] = __dadd_rn(m[l], v);
  }
  if (p.Sd) {
    for (int g = 0; g < p.G; ++g) {
      const double v = p.Sd[(size_t)k * p.G + g];
#pragma unroll
      for (int l = 0; l < kMaxL; ++l)
        if (l == p.hn[g]) m[l] = __dadd_rn(m[l], v);
    }
  }
  for (int l = 0; l < p.L; ++l) p.M[(size_t)k * p.L + l] = m[l];
}

// ------------------------------------------------------------------ solver
struct AssignParams {
  const double* M;   // [n][I][L]
  int32_t* nu;       // [n][I]
  double* value;     // [n]
  uint32_t* status;  // latched AFF_ERR_NO_CONVERGENCE
  int64_t I;
  int L;
  int iters;
  double decay;
  int64_t max_cycles;
};

struct Best {   // a candidate move: larger gain wins, then the lower index
  double gain;
  int64_t idx;
};

__device__ __forceinline__ bool better(const Best& a, const Best& b) {
  return a.gain > b.gain || (a.gain == b.gain && a.idx < b.idx);
}

__device__ __forceinline__ Best warp_best(Best v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Best w{__shfl_down_sync(0xffffffffu, v.gain, o), __shfl_down_sync(0xffffffffu, v.idx, o)};
    if (better(w, v)) v = w;
  }
  return v;
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  return v;
}

// Block-wide reductions in a fixed order (deterministic).
__device__ double block_sum(double v, double* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  v = warp_sum(v);
  if (lane == 0) red[w] = v;
  __syncthreads();
  double t = 0.0;
  if (w == 0) {
    t = warp_sum(lane < kWarps ? red[lane] : 0.0);
    if (lane == 0) red[0] = t;
  }
  __syncthreads();
  t = red[0];
  __syncthreads();
  return t;
}

__device__ Best block_best(Best v, Best* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  v = warp_best(v);
  if (lane == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    Best t = lane < kWarps ? red[lane] : Best{-INFINITY, INT64_MAX};
    t = warp_best(t);
    if (lane == 0) red[0] = t;
  }
  __syncthreads();
  const Best r = red[0];
  __syncthreads();
  return r;
}

struct SolverShared {
  double pi[kMaxL];
  int cnt[kMaxL];
  double red[kWarps];
  Best bred[kWarps];
  double wgain[kMaxL * kMaxL];
  int64_t wk[kMaxL * kMaxL];
  Best pair[kWarps][kMaxL * kMaxL];
  int done;
};

// Best exchange cycle over the L devices from the best single move per
// ordered pair (w[a][b]: gain of moving a neuron from a to b).  Cycles are
// enumerated with their smallest device first; the first maximum wins.
__device__ int best_cycle(const double* w, int L, int* cyc, double* gain) {
  int best_len = 0;
  double best = -INFINITY;
  int path[kMaxL], next[kMaxL];
  bool used[kMaxL];
  for (int s = 0; s < L; ++s) {
    for (int i = 0; i < L; ++i) used[i] = false;
    int depth = 0;
    path[0] = s;
    used[s] = true;
    next[0] = s + 1;
    double acc[kMaxL];
    acc[0] = 0.0;
    while (depth >= 0) {
      if (next[depth] >= L) {
        used[path[depth]] = false;
        --depth;
        continue;
      }
      const int v = next[depth]++;
      if (used[v]) continue;
      const int u = path[depth];
      const double a = acc[depth] + w[u * L + v];
      const double closed = a + w[v * L + s];
      if (closed > best) {
        best = closed;
        best_len = depth + 2;
        for (int i = 0; i <= depth; ++i) cyc[i] = path[i];
        cyc[depth + 1] = v;
      }
      if (depth + 2 < L) {
        ++depth;
        path[depth] = v;
        used[v] = true;
        acc[depth] = a;
        next[depth] = s + 1;
      }
    }
  }
  *gain = best;
  return best_len;
}

__global__ void __launch_bounds__(kAssignThreads, 1) assign_neurons_kernel(AssignParams p) {
  extern __shared__ __align__(16) int32_t s_nu[];  // [I]
  __shared__ SolverShared sh;
  const int tid = threadIdx.x;
  const int L = p.L;
  const int64_t I = p.I;
  const int cap = (int)(I / L);
  const double* M = p.M + (size_t)blockIdx.x * I * L;
  auto m = [&](int64_t k, int l) { return __ldg(M + (size_t)k * L + l); };

  // scale of the problem: mean spread of a row (first dual step) and max |M| (tolerance)
  double spread = 0.0, amax = 0.0;
  for (int64_t k = tid; k < I; k += kAssignThreads) {
    double lo = m(k, 0), hi = lo;
    for (int l = 1; l < L; ++l) {
      const double v = m(k, l);
      lo = fmin(lo, v);
      hi = fmax(hi, v);
    }
    spread += hi - lo;
    amax = fmax(amax, fmax(fabs(lo), fabs(hi)));
  }
  spread = block_sum(spread, sh.red) / (double)I;
  {
    Best b = block_best(Best{amax, 0}, sh.bred);
    amax = b.gain;
  }
  const double tol = 64.0 * DBL_EPSILON * amax;

  // 1. dual ascent on the device offsets pi: every neuron takes its best
  //    device at the current prices; over-subscribed devices get dearer.
  if (tid < L) sh.pi[tid] = 0.0;
  __syncthreads();
  double step = spread;
  for (int it = 0; it < p.iters; ++it) {
    if (tid < L) sh.cnt[tid] = 0;
    __syncthreads();
    for (int64_t k = tid; k < I; k += kAssignThreads) {
      int bl = 0;
      double bv = m(k, 0) - sh.pi[0];
      for (int l = 1; l < L; ++l) {
        const double v = m(k, l) - sh.pi[l];
        if (v > bv) { bv = v; bl = l; }
      }
      atomicAdd(&sh.cnt[bl], 1);
    }
    __syncthreads();
    if (tid < L) sh.pi[tid] += step * (double)(sh.cnt[tid] - cap) / (double)cap;
    step *= p.decay;
    __syncthreads();
  }

  // 2. the map at the final prices
  if (tid < L) sh.cnt[tid] = 0;
  __syncthreads();
  for (int64_t k = tid; k < I; k += kAssignThreads) {
    int bl = 0;
    double bv = m(k, 0) - sh.pi[0];
    for (int l = 1; l < L; ++l) {
      const double v = m(k, l) - sh.pi[l];
      if (v > bv) { bv = v; bl = l; }
    }
    s_nu[k] = bl;
    atomicAdd(&sh.cnt[bl], 1);
  }
  __syncthreads();

  // 3. fix-up: while a device is over capacity, make the cheapest single move
  //    from an over-full device to an under-full one.
  for (int64_t guard = 0; guard <= I; ++guard) {
    bool over = false;
    for (int l = 0; l < L; ++l) over |= sh.cnt[l] > cap;
    if (!over) break;
    Best b{-INFINITY, INT64_MAX};
    for (int64_t k = tid; k < I; k += kAssignThreads) {
      const int a = s_nu[k];
      if (sh.cnt[a] <= cap) continue;
      for (int l = 0; l < L; ++l) {
        if (sh.cnt[l] >= cap) continue;
        const Best c{m(k, l) - m(k, a), k * kMaxL + l};
        if (better(c, b)) b = c;
      }
    }
    b = block_best(b, sh.bred);
    if (tid == 0 && b.idx != INT64_MAX) {
      const int64_t k = b.idx / kMaxL;
      const int to = (int)(b.idx % kMaxL);
      sh.cnt[s_nu[k]]--;
      sh.cnt[to]++;
      s_nu[k] = to;
    }
    __syncthreads();
  }

  // 4. exchange cycles until none gains
  const int lane = tid & 31, wid = tid >> 5;
  int64_t c = 0;
  for (; c < p.max_cycles; ++c) {
    Best loc[kMaxL * kMaxL];
#pragma unroll
    for (int i = 0; i < kMaxL * kMaxL; ++i) loc[i] = Best{-INFINITY, INT64_MAX};
    for (int64_t k = tid; k < I; k += kAssignThreads) {
      const int a = s_nu[k];
      const double base = m(k, a);
      for (int b = 0; b < L; ++b) {
        if (b == a) continue;
        const Best cand{m(k, b) - base, k};
        if (better(cand, loc[a * kMaxL + b])) loc[a * kMaxL + b] = cand;
      }
    }
    for (int a = 0; a < L; ++a)
      for (int b = 0; b < L; ++b) {
        Best v = warp_best(loc[a * kMaxL + b]);
        if (lane == 0) sh.pair[wid][a * L + b] = v;
      }
    __syncthreads();
    if (tid < L * L) {
      Best v{-INFINITY, INT64_MAX};
      for (int w = 0; w < kWarps; ++w)
        if (better(sh.pair[w][tid], v)) v = sh.pair[w][tid];
      sh.wgain[tid] = (tid / L == tid % L) ? -INFINITY : v.gain;
      sh.wk[tid] = v.idx;
    }
    __syncthreads();
    if (tid == 0) {
      int cyc[kMaxL];
      double g = 0.0;
      const int len = best_cycle(sh.wgain, L, cyc, &g);
      if (len < 2 || !(g > tol)) {
        sh.done = 1;
      } else {
        sh.done = 0;
        for (int i = 0; i < len; ++i) {
          const int a = cyc[i], b = cyc[(i + 1) % len];
          s_nu[sh.wk[a * L + b]] = b;
        }
      }
    }
    __syncthreads();
    if (sh.done) break;
  }
  if (c >= p.max_cycles && tid == 0) atomicOr(p.status, (uint32_t)AFF_ERR_NO_CONVERGENCE);

  // 5. the map and its value
  double v = 0.0;
  for (int64_t k = tid; k < I; k += kAssignThreads) {
    const int l = s_nu[k];
    p.nu[(size_t)blockIdx.x * I + k] = l;
    v += m(k, l);
  }
  v = block_sum(v, sh.red);
  if (tid == 0) p.value[blockIdx.x] = v;
}

bool aligned8(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 7u) == 0; }

aff_status check_assign_shape(int64_t I, int32_t L) {
  if (L < 1 || L > kMaxL || I < L || I % L) return AFF_ERR_UNSUPPORTED_SHAPE;
  if (I > kMaxNeurons) return AFF_ERR_UNSUPPORTED_SHAPE;
  return AFF_OK;
}

void fill_opts(const aff_assign_opts* o, int64_t I, AssignParams& p) {
  p.iters = (o && o->dual_iters > 0) ? o->dual_iters : 300;
  p.decay = (o && o->dual_decay > 0.0 && o->dual_decay <= 1.0) ? o->dual_decay : 0.98;
  p.max_cycles = (o && o->max_cycles > 0) ? o->max_cycles : 64 * I;
}

aff_status launch_gain(const double* Su, const double* Sd, const int32_t* h, const int32_t* hn, int G, int64_t I,
                       int L, double* M, cudaStream_t s) {
  GainParams gp{};
  gp.Su = Su;
  gp.Sd = Sd;
  gp.M = M;
  gp.I = I;
  gp.G = G;
  gp.L = L;
  for (int g = 0; g < G; ++g) {
    gp.h[g] = (int8_t)h[g];
    gp.hn[g] = Sd ? (int8_t)hn[g] : 0;
  }
  const int threads = 256;
  neuron_gain_kernel<<<(unsigned)((I + threads - 1) / threads), threads, 0, s>>>(gp);
  AFF_CUDA(cudaGetLastError());
  return AFF_OK;
}

aff_status launch_assign(const double* M, int n_layers, int64_t I, int L, const aff_assign_opts* opts, int32_t* nu,
                         double* value, uint32_t* status, cudaStream_t s) {
  AssignParams ap{};
  ap.M = M;
  ap.nu = nu;
  ap.value = value;
  ap.status = status;
  ap.I = I;
  ap.L = L;
  fill_opts(opts, I, ap);
  const size_t smem = (size_t)I * sizeof(int32_t);
  // the opt-in is per device, so it is set on every call (a cheap host call)
  AFF_CUDA(cudaFuncSetAttribute(assign_neurons_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(kMaxNeurons * sizeof(int32_t))));
  assign_neurons_kernel<<<n_layers, kAssignThreads, smem, s>>>(ap);
  AFF_CUDA(cudaGetLastError());
  return AFF_OK;
}

bool maps_ok(const int32_t* m, int64_t n, int L) {
  for (int64_t i = 0; i < n; ++i)
    if (m[i] < 0 || m[i] >= L) return false;
  return true;
}

bool balanced(const int32_t* m, int64_t n, int L) {
  std::vector<int64_t> c(L, 0);
  for (int64_t i = 0; i < n; ++i) c[m[i]]++;
  for (int l = 0; l < L; ++l)
    if (c[l] != n / L) return false;
  return true;
}

struct LayoutWs {
  size_t status, up, down, M, nu, value, total;
};

LayoutWs layout_ws(int32_t N, int32_t G, int64_t I, int32_t L) {
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  LayoutWs w{};
  size_t o = 0;
  w.status = o; o += 256;
  w.up = o; o = up(o + (size_t)N * G * I * sizeof(double));
  w.down = o; o = up(o + (size_t)(N > 1 ? N - 1 : 0) * I * G * sizeof(double));
  w.M = o; o = up(o + (size_t)N * I * L * sizeof(double));
  w.nu = o; o = up(o + (size_t)N * I * sizeof(int32_t));
  w.value = o; o = up(o + (size_t)N * sizeof(double));
  w.total = o;
  return w;
}

}  // namespace
}  // namespace aff

using namespace aff;

extern "C" {

aff_status affinity_neuron_gain(const double* Shat_up_i, const double* Shat_down_i, const int32_t* h_i,
                                const int32_t* h_next, int32_t G, int64_t I, int32_t L, double* M_out,
                                aff_stream_t stream) {
  if (!Shat_up_i || !h_i || !M_out || G < 1 || G > kMaxG || I < 1) return AFF_ERR_INVALID_ARG;
  if ((Shat_down_i == nullptr) != (h_next == nullptr)) return AFF_ERR_INVALID_ARG;
  if (L < 1 || L > kMaxL) return AFF_ERR_UNSUPPORTED_SHAPE;
  if (!maps_ok(h_i, G, L) || (h_next && !maps_ok(h_next, G, L))) return AFF_ERR_INVALID_ARG;
  if (!aligned8(Shat_up_i) || (Shat_down_i && !aligned8(Shat_down_i)) || !aligned8(M_out)) return AFF_ERR_ALIGNMENT;
  int sms = 0;
  aff_status st = check_device(&sms);
  if (st != AFF_OK) return st;
  return launch_gain(Shat_up_i, Shat_down_i, h_i, h_next, G, I, L, M_out, reinterpret_cast<cudaStream_t>(stream));
}

aff_status affinity_assign_neurons(const double* M, int32_t n_layers, int64_t I, int32_t L,
                                   const aff_assign_opts* opts, int32_t* nu_out, double* value_out, void* workspace,
                                   size_t workspace_bytes, aff_stream_t stream) {
  if (!M || !nu_out || !value_out || n_layers < 1) return AFF_ERR_INVALID_ARG;
  aff_status st = check_assign_shape(I, L);
  if (st != AFF_OK) return st;
  if (!workspace || workspace_bytes < 256 || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return AFF_ERR_WORKSPACE;
  if (!aligned8(M) || !aligned8(value_out) || (reinterpret_cast<uintptr_t>(nu_out) & 3u)) return AFF_ERR_ALIGNMENT;
  int sms = 0;
  if ((st = check_device(&sms)) != AFF_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* status = reinterpret_cast<uint32_t*>(workspace);
  AFF_CUDA(cudaMemsetAsync(status, 0, 4, s));
  return launch_assign(M, n_layers, I, L, opts, nu_out, value_out, status, s);
}

aff_status affinity_layout_workspace_size(int32_t N, int32_t G, int64_t I, int32_t L, size_t* bytes) {
  if (!bytes || N < 1 || G < 1 || G > kMaxG) return AFF_ERR_INVALID_ARG;
  aff_status st = check_assign_shape(I, L);
  if (st != AFF_OK) return st;
  if (G % L) return AFF_ERR_UNSUPPORTED_SHAPE;
  *bytes = layout_ws(N, G, I, L).total;
  return AFF_OK;
}

aff_status affinity_optimise_layout(const double* Shat_up, const double* Shat_down, int32_t N, int32_t G, int64_t I,
                                    int32_t L, const aff_layout_opts* opts, int32_t* h, int32_t* nu, double* J_out,
                                    int32_t* sweeps_out, void* workspace, size_t workspace_bytes,
                                    aff_stream_t stream) {
  if (!Shat_up || !h || !nu || !J_out || N < 1 || G < 1 || G > kMaxG) return AFF_ERR_INVALID_ARG;
  if (N > 1 && !Shat_down) return AFF_ERR_INVALID_ARG;
  aff_status st = check_assign_shape(I, L);
  if (st != AFF_OK) return st;
  if (G % L) return AFF_ERR_UNSUPPORTED_SHAPE;
  if (!maps_ok(h, (int64_t)N * G, L) || !maps_ok(nu, (int64_t)N * I, L)) return AFF_ERR_INVALID_ARG;
  for (int i = 0; i < N; ++i)
    if (!balanced(h + (size_t)i * G, G, L) || !balanced(nu + (size_t)i * I, I, L)) return AFF_ERR_INVALID_ARG;
  const LayoutWs W = layout_ws(N, G, I, L);
  if (!workspace || workspace_bytes < W.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return AFF_ERR_WORKSPACE;
  int sms = 0;
  if ((st = check_device(&sms)) != AFF_OK) return st;

  const int max_sweeps = (opts && opts->max_sweeps > 0) ? opts->max_sweeps : 16;
  const bool move_heads = !(opts && opts->freeze_heads);
  const bool move_neurons = !(opts && opts->freeze_neurons);
  const bool minimise = opts && opts->minimise;
  const uint8_t* mask = opts ? opts->layer_mask : nullptr;
  const aff_assign_opts* aopts = opts ? &opts->assign : nullptr;
  const double sign = minimise ? -1.0 : 1.0;

  // signed copies (minimising J maximises -J) on the host and the device
  const size_t nu_up = (size_t)N * G * I, nu_dn = (size_t)(N - 1) * I * G;
  std::vector<double> up(nu_up), dn(nu_dn);
  for (size_t i = 0; i < nu_up; ++i) up[i] = sign * Shat_up[i];
  for (size_t i = 0; i < nu_dn; ++i) dn[i] = sign * Shat_down[i];
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  double* d_up = reinterpret_cast<double*>(ws + W.up);
  double* d_dn = reinterpret_cast<double*>(ws + W.down);
  double* d_M = reinterpret_cast<double*>(ws + W.M);
  int32_t* d_nu = reinterpret_cast<int32_t*>(ws + W.nu);
  double* d_val = reinterpret_cast<double*>(ws + W.value);
  uint32_t* d_status = reinterpret_cast<uint32_t*>(ws + W.status);
  AFF_CUDA(cudaMemsetAsync(d_status, 0, 4, s));
  AFF_CUDA(cudaMemcpyAsync(d_up, up.data(), nu_up * sizeof(double), cudaMemcpyHostToDevice, s));
  if (nu_dn) AFF_CUDA(cudaMemcpyAsync(d_dn, dn.data(), nu_dn * sizeof(double), cudaMemcpyHostToDevice, s));

  double J = 0.0;
  if ((st = affinity_objective(up.data(), N > 1 ? dn.data() : nullptr, h, nu, N, G, I, &J)) != AFF_OK) return st;
  std::vector<int32_t> h_new((size_t)N * G), nu_new((size_t)N * I);
  std::vector<double> C((size_t)G * L);
  int sweeps = 0;
  while (sweeps < max_sweeps) {
    ++sweeps;
    std::memcpy(h_new.data(), h, h_new.size() * sizeof(int32_t));
    std::memcpy(nu_new.data(), nu, nu_new.size() * sizeof(int32_t));
    if (move_neurons) {
      // every layer's neuron step at once: M_i needs only h_i and h_{i+1}
      for (int i = 0; i < N; ++i) {
        const bool down = i + 1 < N;
        if ((st = launch_gain(d_up + (size_t)i * G * I, down ? d_dn + (size_t)i * I * G : nullptr,
                              h + (size_t)i * G, down ? h + (size_t)(i + 1) * G : nullptr, G, I, L,
                              d_M + (size_t)i * I * L, s)) != AFF_OK)
          return st;
      }
      if ((st = launch_assign(d_M, N, I, L, aopts, d_nu, d_val, d_status, s)) != AFF_OK) return st;
      AFF_CUDA(cudaMemcpyAsync(nu_new.data(), d_nu, nu_new.size() * sizeof(int32_t), cudaMemcpyDeviceToHost, s));
      uint32_t dev_status = 0;
      AFF_CUDA(cudaMemcpyAsync(&dev_status, d_status, 4, cudaMemcpyDeviceToHost, s));
      AFF_CUDA(cudaStreamSynchronize(s));
      if (dev_status) return static_cast<aff_status>(dev_status);
      if (mask)
        for (int i = 0; i < N; ++i)
          if (!mask[i]) std::memcpy(&nu_new[(size_t)i * I], nu + (size_t)i * I, I * sizeof(int32_t));
    }
    if (move_heads) {
      // every layer's head step given the new neuron maps: h_i needs nu_{i-1} and nu_i
      for (int i = 0; i < N; ++i) {
        if (mask && !mask[i]) continue;
        const double* Sd = i > 0 ? dn.data() + (size_t)(i - 1) * I * G : nullptr;
        const int32_t* np = i > 0 ? nu_new.data() + (size_t)(i - 1) * I : nullptr;
        if ((st = affinity_group_gain(up.data() + (size_t)i * G * I, nu_new.data() + (size_t)i * I, Sd, np, G, I, L,
                                      C.data())) != AFF_OK)
          return st;
        int64_t count = 0, best = 0;
        if ((st = affinity_score_partitions(C.data(), G, L, nullptr, &count, &best, h_new.data() + (size_t)i * G)) !=
            AFF_OK)
          return st;
      }
    }
    double J_new = 0.0;
    if ((st = affinity_objective(up.data(), N > 1 ? dn.data() : nullptr, h_new.data(), nu_new.data(), N, G, I,
                                 &J_new)) != AFF_OK)
      return st;
    // each step is optimal given the others, so J never falls; stop once it stalls
    const bool gained = J_new > J + 1e-12 * std::fabs(J);
    if (J_new >= J) {
      std::memcpy(h, h_new.data(), h_new.size() * sizeof(int32_t));
      std::memcpy(nu, nu_new.data(), nu_new.size() * sizeof(int32_t));
      J = J_new;
    }
    if (!gained) break;
  }
  *J_out = sign * J;
  if (sweeps_out) *sweeps_out = sweeps;
  return AFF_OK;
}

}  // extern "C"
