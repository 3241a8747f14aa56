// aux_kernels.cu -- the memory-bound and small kernels around the tcgen05
// tile kernel: operand staging in fp16, the deterministic cross-unit
// reductions, the down-edge finishing steps, and the fp32 CUDA-core path.
// Paper: "Affinity-Aware Sharding for Delayed Tensor Parallelism", §3
// "Affinity scores" (eq. 5 and the FO / ADD / down definitions after it).
#include "aux_kernels.cuh"
#include "launch.cuh"
#include "scales.cuh"
#include "sm103_primitives.cuh"

#include <cuda_fp16.h>

namespace aff {

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ __half to_h(float v, bool& bad) {
  if (!(fabsf(v) <= 65504.f)) bad = true;
  return __float2half_rn(v);
}

// fp16 of v, its magnitude folded into m (fp32 bits) for the staging maxima.
__device__ __forceinline__ __half to_h_max(float v, uint32_t& m) {
  m = max(m, __float_as_uint(fabsf(v)));
  return __float2half_rn(v);
}

// ---------------------------------------------------------------- token rows
// One warp per token: r_t = sqrt(mean_d x_td^2 + eps); n16 = gamma*x/r (the
// FFN's normalised input) times 2^e_n and a16 = a/r (so that the head
// contraction with the folded matrices yields p_h.w directly), both rounded to
// fp16, and 1/r.  e_n comes from max|gamma| (every block finds the same value;
// block 0 records it).  a16 is staged unscaled while the largest |a/r| is
// recorded; restage_a_kernel rescales it when that maximum calls for it.
__global__ void prep_tokens_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ a,
                                   const uint16_t* __restrict__ gamma, __half* __restrict__ n16,
                                   __half* __restrict__ a16, float* __restrict__ inv_r, int T, int D, int HD,
                                   float eps, uint32_t* status, DevScales* sc) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int n_warps = (gridDim.x * blockDim.x) >> 5;
  __shared__ uint32_t gmax_s;
  if (threadIdx.x == 0) gmax_s = 0u;
  __syncthreads();
  uint32_t gm = 0u;   // |gamma| as fp32 bits: the bf16 magnitude bits, shifted
  for (int v = threadIdx.x; v < D; v += blockDim.x) gm = max(gm, (uint32_t)(gamma[v] & 0x7FFFu) << 16);
  gm = __reduce_max_sync(0xffffffffu, gm);
  if (lane == 0) atomicMax(&gmax_s, gm);
  __syncthreads();
  DevScales loc{};
  loc.gmax = gmax_s;
  if (blockIdx.x == 0 && threadIdx.x == 0) sc->gmax = gmax_s;
  const float fn = pow2f(scale_exps(loc, D).e_n);
  bool bad = false;
  uint32_t am = 0u;   // largest |a / r| this thread staged (fp32 bits)
  for (int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; warp < T; warp += n_warps) {
  const size_t t = (size_t)warp;
  const uint4* xr = reinterpret_cast<const uint4*>(x + t * D);
  float ss = 0.f;
  for (int v = lane; v < D / 8; v += 32) {
    uint4 q = xr[v];
    const uint16_t* e = reinterpret_cast<const uint16_t*>(&q);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float f = bf2f(e[i]);
      ss = fmaf(f, f, ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float ir = rsqrtf(ss / (float)D + eps);
  if (lane == 0 && inv_r) inv_r[t] = ir;
  if (n16) {
    const float irn = ir * fn;
    const uint4* gr = reinterpret_cast<const uint4*>(gamma);
    uint4* nr = reinterpret_cast<uint4*>(n16 + t * D);
    for (int v = lane; v < D / 8; v += 32) {
      uint4 q = xr[v], g = gr[v];
      const uint16_t* e = reinterpret_cast<const uint16_t*>(&q);
      const uint16_t* ge = reinterpret_cast<const uint16_t*>(&g);
      __align__(16) __half o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = to_h(bf2f(ge[i]) * (bf2f(e[i]) * irn), bad);
      nr[v] = *reinterpret_cast<uint4*>(o);
    }
  }
  if (a16) {
    const uint4* ar = reinterpret_cast<const uint4*>(a + t * HD);
    uint4* orow = reinterpret_cast<uint4*>(a16 + t * HD);
    for (int v = lane; v < HD / 8; v += 32) {
      uint4 q = ar[v];
      const uint16_t* e = reinterpret_cast<const uint16_t*>(&q);
      __align__(16) __half o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float f = bf2f(e[i]) * ir;
        am = max(am, __float_as_uint(fabsf(f)));
        o[i] = __float2half_rn(f);
      }
      orow[v] = *reinterpret_cast<uint4*>(o);
    }
  }
  }
  if (a16) {
    am = __reduce_max_sync(0xffffffffu, am);
    if (lane == 0 && am) atomicMax(&sc->amax, am);
  }
  if (bad) latch_status(status, kStatusRange);
}

// a16 = fp16(a / r * 2^e_a) for every token, when the largest |a/r| recorded by
// prep_tokens_kernel lies outside [2^-6, 2^15) (e_a != 0); otherwise nothing to
// do.  A non-finite maximum (a non-finite input) latches AFF_ERR_RANGE.
__global__ void restage_a_kernel(const uint16_t* __restrict__ a, const float* __restrict__ inv_r,
                                 __half* __restrict__ a16, int T, int HD, const DevScales* __restrict__ sc,
                                 uint32_t* status) {
  pdl_enter();
  const float am = bits_f(sc->amax);
  if (!(am <= 3.4e38f)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) latch_status(status, kStatusRange);
    return;
  }
  const int e = scale_exp_act(am);
  if (e == 0) return;
  const float f = pow2f(e);
  const size_t n8 = (size_t)T * HD / 8;
  for (size_t v = blockIdx.x * (size_t)blockDim.x + threadIdx.x; v < n8; v += (size_t)gridDim.x * blockDim.x) {
    const size_t t = v * 8 / HD;
    const float irf = inv_r[t] * f;
    const uint4 q = *reinterpret_cast<const uint4*>(a + v * 8);
    const uint16_t* e8 = reinterpret_cast<const uint16_t*>(&q);
    __align__(16) __half o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = __float2half_rn(bf2f(e8[i]) * irf);
    *reinterpret_cast<uint4*>(a16 + v * 8) = *reinterpret_cast<uint4*>(o);
  }
}

// W16 = fp16 copy of Wg and Wu, I_pad neurons (zero rows past I), in groups of 16
// neurons: their 16 gate rows, then their 16 up rows ([I_pad / 16][2][16][D]).
// One warp per row, staged unscaled while the largest magnitude is recorded in
// sc->wmax; weight_restage_kernel rescales when that maximum calls for it.
__device__ __forceinline__ void stage_w16_rows(const uint16_t* __restrict__ Wg, const uint16_t* __restrict__ Wu,
                                               __half* __restrict__ W16, int I, int I_pad, int D, int warp0,
                                               int nwarps, float f, uint32_t& m) {
  const int lane = threadIdx.x & 31;
  const int D8 = D / 8;
  for (int r = warp0; r < 2 * I_pad; r += nwarps) {
    // row r: neuron group r / 32, gate (0) or up (1) row, neuron 16 * (r / 32) + r % 16
    const int blk = (r >> 4) & 1, k = (r >> 5) * 16 + (r & 15);
    const uint4* src = reinterpret_cast<const uint4*>((blk == 0 ? Wg : Wu) + (size_t)k * D);
    uint4* dst = reinterpret_cast<uint4*>(W16 + (size_t)r * D);
    // four 16-byte loads of the row in flight per lane, then their conversion
    for (int c0 = lane; c0 < D8; c0 += 4 * 32) {
      uint4 q[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = c0 + 32 * j;
        q[j] = (k < I && c < D8) ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = c0 + 32 * j;
        if (c < D8) {
          __align__(16) __half o[8];
          const uint16_t* e = reinterpret_cast<const uint16_t*>(&q[j]);
#pragma unroll
          for (int i = 0; i < 8; ++i) o[i] = to_h_max(bf2f(e[i]) * f, m);
          dst[c] = *reinterpret_cast<uint4*>(o);
        }
      }
    }
  }
}

__global__ void __launch_bounds__(256) prep_gate_up_kernel(const uint16_t* __restrict__ Wg,
                                                           const uint16_t* __restrict__ Wu,
                                                           __half* __restrict__ W16, int I, int I_pad, int D,
                                                           DevScales* sc) {
  pdl_enter();
  uint32_t m = 0u;
  stage_w16_rows(Wg, Wu, W16, I, I_pad, D, (blockIdx.x * blockDim.x + threadIdx.x) >> 5,
                 (gridDim.x * blockDim.x) >> 5, 1.0f, m);
  m = __reduce_max_sync(0xffffffffu, m);
  if ((threadIdx.x & 31) == 0 && m) atomicMax(&sc->wmax, m);
}

// GWo16[n][part][d] for part 0/1 = fp16 hi / lo of gamma_d * Wo[d][n] * f (a
// transposed, split copy through 64 x 64 shared-memory tiles, 16-byte loads and
// stores: hi + lo carries ~22 significant bits of the exact fp32 product); 256
// threads, grid-stride over tiles starting at tile0.  D and HD are multiples of
// 8, so an 8-element chunk is wholly inside or wholly outside.  Folds
// max |gamma_d Wo[d][n]| (before f) into gm and max |Wo[d][n]| into om.
__device__ __forceinline__ void stage_gwo_tiles(const uint16_t* __restrict__ Wo, const uint16_t* __restrict__ gamma,
                                                __half* __restrict__ GWo16, int D, int HD, int tile0, int ntiles_step,
                                                float f, uint32_t& gm, uint32_t& om) {
  __shared__ float tile[64][65];   // [d][n], padded: column reads hit distinct banks but for 2-way
  const int tn = (HD + 63) / 64, td = (D + 63) / 64;
  for (int tt = tile0; tt < tn * td; tt += ntiles_step) {
    const int d0 = (tt / tn) * 64, n0 = (tt % tn) * 64;
    __syncthreads();
    // 64 rows d x 8 chunks of 8 columns n: both of a thread's loads issued first
    uint4 q[2];
    uint16_t gb[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int it = threadIdx.x + 256 * u;
      const int d = d0 + (it >> 3), n = n0 + (it & 7) * 8;
      const bool in = d < D && n < HD;
      q[u] = in ? __ldg(reinterpret_cast<const uint4*>(Wo + (size_t)d * HD + n)) : make_uint4(0u, 0u, 0u, 0u);
      gb[u] = in ? gamma[d] : (uint16_t)0;
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int it = threadIdx.x + 256 * u;
      const int i = it >> 3, c = (it & 7) * 8;
      const uint16_t* e = reinterpret_cast<const uint16_t*>(&q[u]);
      const float g = bf2f(gb[u]);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float w = bf2f(e[j]);
        om = max(om, __float_as_uint(fabsf(w)));
        const float gw = g * w;
        gm = max(gm, __float_as_uint(fabsf(gw)));
        tile[i][c + j] = gw * f;
      }
    }
    __syncthreads();
    // 64 rows n x 8 chunks of 8 columns d, hi and lo
    for (int it = threadIdx.x; it < 512; it += 256) {
      const int i = it >> 3, c = (it & 7) * 8;
      const int n = n0 + i, d = d0 + c;
      if (n < HD && d < D) {
        __align__(16) __half hi[8];
        __align__(16) __half lo[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float v = tile[c + j][i];
          hi[j] = __float2half_rn(v);
          lo[j] = __float2half_rn(v - __half2float(hi[j]));
        }
        *reinterpret_cast<uint4*>(GWo16 + ((size_t)n * 2 + 0) * D + d) = *reinterpret_cast<const uint4*>(hi);
        *reinterpret_cast<uint4*>(GWo16 + ((size_t)n * 2 + 1) * D + d) = *reinterpret_cast<const uint4*>(lo);
      }
    }
  }
}

// The weight staging of the up pass in one launch, unscaled, recording the maxima
// of DevScales: blockIdx.y == 0 stages W16, blockIdx.y == 1 stages GWo16.  Both
// parts grid-stride.
__global__ void __launch_bounds__(256) weight_stage_kernel(const uint16_t* __restrict__ Wg,
                                                           const uint16_t* __restrict__ Wu, __half* __restrict__ W16,
                                                           int I, int I_pad, int D, const uint16_t* __restrict__ Wo,
                                                           const uint16_t* __restrict__ gamma,
                                                           __half* __restrict__ GWo16, int HD, DevScales* sc) {
  pdl_enter();
  if (blockIdx.y == 0) {
    uint32_t m = 0u;
    stage_w16_rows(Wg, Wu, W16, I, I_pad, D, blockIdx.x * 8 + (threadIdx.x >> 5), gridDim.x * 8, 1.0f, m);
    m = __reduce_max_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0 && m) atomicMax(&sc->wmax, m);
  } else {
    uint32_t gm = 0u, om = 0u;
    stage_gwo_tiles(Wo, gamma, GWo16, D, HD, blockIdx.x, gridDim.x, 1.0f, gm, om);
    gm = __reduce_max_sync(0xffffffffu, gm);
    om = __reduce_max_sync(0xffffffffu, om);
    if ((threadIdx.x & 31) == 0) {
      if (gm) atomicMax(&sc->gwmax, gm);
      if (om) atomicMax(&sc->womax, om);
    }
  }
}

// The weights staged again at their power-of-two scales (scales.cuh) when the
// recorded maxima call for it; otherwise every block returns at once.  y = 0:
// W16 = W 2^e_w; y = 1: GWo16 = gamma Wo^T 2^e_g (when given); y = 2: Wo16 =
// Wo 2^e_o (when given: the leave-one-out pass).  A non-finite maximum (a
// non-finite weight) latches AFF_ERR_RANGE.
__global__ void __launch_bounds__(256) weight_restage_kernel(const uint16_t* __restrict__ Wg,
                                                             const uint16_t* __restrict__ Wu,
                                                             __half* __restrict__ W16, int I, int I_pad, int D,
                                                             const uint16_t* __restrict__ Wo,
                                                             const uint16_t* __restrict__ gamma,
                                                             __half* __restrict__ GWo16, __half* __restrict__ Wo16,
                                                             int HD, DevScales* sc, uint32_t* status) {
  pdl_enter();
  if (blockIdx.y == 1 && GWo16 == nullptr) return;
  if (blockIdx.y == 2 && Wo16 == nullptr) return;
  const float m = bits_f(blockIdx.y == 0 ? sc->wmax : (blockIdx.y == 1 ? sc->gwmax : sc->womax));
  if (!(m <= 3.4e38f)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) latch_status(status, kStatusRange);
    return;
  }
  const int e = scale_exp_act(m);
  if (e == 0) return;
  const float f = pow2f(e);
  uint32_t m1 = 0u, m2 = 0u;   // maxima seen again here (the recorded ones stay)
  if (blockIdx.y == 0) {
    stage_w16_rows(Wg, Wu, W16, I, I_pad, D, blockIdx.x * 8 + (threadIdx.x >> 5), gridDim.x * 8, f, m1);
  } else if (blockIdx.y == 1) {
    stage_gwo_tiles(Wo, gamma, GWo16, D, HD, blockIdx.x, gridDim.x, f, m1, m2);
  } else {
    const size_t n8 = (size_t)D * HD / 8;
    for (size_t v = blockIdx.x * (size_t)blockDim.x + threadIdx.x; v < n8; v += (size_t)gridDim.x * blockDim.x) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(Wo) + v);
      const uint16_t* e8 = reinterpret_cast<const uint16_t*>(&q);
      __align__(16) __half o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = __float2half_rn(bf2f(e8[i]) * f);
      reinterpret_cast<uint4*>(Wo16)[v] = *reinterpret_cast<uint4*>(o);
    }
  }
}

// wdn[k] = ||w^d_k||^2 = sum_d Wd[d][k]^2 (fp32; fixed order: 8 row phases, then in order).
__global__ void wd_colnorm_kernel(const uint16_t* __restrict__ Wd, float* __restrict__ wdn, int D, int I, int I_pad) {
  pdl_enter();
  __shared__ float part[8][33];
  const int k = blockIdx.x * 32 + threadIdx.x;
  float s = 0.f;
  if (k < I)
    for (int d = threadIdx.y; d < D; d += 8) {
      const float v = bf2f(Wd[(size_t)d * I + k]);
      s = fmaf(v, v, s);
    }
  part[threadIdx.y][threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.y == 0 && k < I_pad) {
    float t = 0.f;
    for (int i = 0; i < 8; ++i) t += part[i][threadIdx.x];
    wdn[k] = (k < I) ? t : 0.f;
  }
}

// fp32 twin of wd_colnorm_kernel for the fp32 path.
__global__ void wd_colnorm_f32_kernel(const float* __restrict__ Wd, float* __restrict__ wdn, int D, int I) {
  __shared__ float part[8][33];
  const int k = blockIdx.x * 32 + threadIdx.x;
  float s = 0.f;
  if (k < I)
    for (int d = threadIdx.y; d < D; d += 8) s = fmaf(Wd[(size_t)d * I + k], Wd[(size_t)d * I + k], s);
  part[threadIdx.y][threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.y == 0 && k < I) {
    float t = 0.f;
    for (int i = 0; i < 8; ++i) t += part[i][threadIdx.x];
    wdn[k] = t;
  }
}

// ---------------------------------------------------------------- reductions
// S_head_d[h][k] = sum over chunks and halves of partial[c][hf][h][k] in a fixed
// order: fp32 sums over 8 interleaved chunk phases, then the phases in fp64
// (fp64 arithmetic is slow on this part, so it is kept to the last level).
__global__ void reduce_partials_kernel(const float* __restrict__ partial, double* __restrict__ out, int n_chunks,
                                       int halves, int H, int I_pad) {
  __shared__ double part[8][33];
  const int k = blockIdx.x * 32 + threadIdx.x;
  const int h = blockIdx.y;
  float s = 0.f;   // fp32 within a phase (at most n_chunks/8 terms), fp64 across the 8 phases
  if (k < I_pad)
    for (int c = threadIdx.y; c < n_chunks; c += 8)
      for (int hf = 0; hf < halves; ++hf) s += partial[((size_t)(c * halves + hf) * H + h) * I_pad + k];
  part[threadIdx.y][threadIdx.x] = (double)s;
  __syncthreads();
  if (threadIdx.y == 0 && k < I_pad) {
    double t = 0.0;
    for (int i = 0; i < 8; ++i) t += part[i][threadIdx.x];
    out[(size_t)h * I_pad + k] = t;
  }
}

// Same reduction, four neurons per thread with 16-byte loads (I_pad % 128 == 0).
__global__ void reduce_partials4_kernel(const float* __restrict__ partial, double* __restrict__ out, int n_chunks,
                                        int halves, int H, int I_pad) {
  __shared__ double part[8][32][4];
  const int k = blockIdx.x * 128 + threadIdx.x * 4;
  const int h = blockIdx.y;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int c = threadIdx.y; c < n_chunks; c += 8)
    for (int hf = 0; hf < halves; ++hf) {
      const float4 v = *reinterpret_cast<const float4*>(partial + ((size_t)(c * halves + hf) * H + h) * I_pad + k);
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
  part[threadIdx.y][threadIdx.x][0] = s.x;
  part[threadIdx.y][threadIdx.x][1] = s.y;
  part[threadIdx.y][threadIdx.x][2] = s.z;
  part[threadIdx.y][threadIdx.x][3] = s.w;
  __syncthreads();
  if (threadIdx.y == 0) {
    for (int e = 0; e < 4; ++e) {
      double t = 0.0;
      for (int i = 0; i < 8; ++i) t += part[i][threadIdx.x][e];
      out[(size_t)h * I_pad + k + e] = t;
    }
  }
}

// The chunk partial sums of one KV group's heads, reduced and finalised in one
// pass: block = 64 neurons x one group, 512 threads.  The partial sums are laid
// out [H][I_pad / 64][n_chunks][groups][64], so each (head, 64-neuron block) is
// one contiguous run of n_chunks * groups rows of 64 floats.  Thread t reads the
// 4 neurons 4 (t % 16).. of rows ph, ph + P, ... (16-byte loads; a warp reads 512
// contiguous bytes); the 32 row phases t / 16 are split among the group's heads R
// at a time (R = min(H/G, 32), P = 32 / R phases a head), so that the loads of R
// heads are in flight together.  Each phase sums its rows in fp32 in order; the
// phases are added in fp64, in order, and
//   S_head[h][k] = sum / T (x ||w^d_k||^2 for FO),  S_up[g][k] = sum_{h in g} S_head[h][k]
// (heads in order).  Needs I_pad % 64 == 0.
template <int GROUPS>
__global__ void __launch_bounds__(512, 3) reduce_finalize_kernel(const float* __restrict__ partial,
                                                              const float* __restrict__ wdn, int fo, int n_chunks,
                                                              int T, int H, int G, int I, int I_pad,
                                                              float* __restrict__ S_out, float* __restrict__ S_head_out,
                                                              const DevScales* __restrict__ sc, int D) {
  pdl_enter();
  // the partial sums carry the head operands' 2^2(e_m + e_a) (scales.cuh)
  const ScaleExps ex = scale_exps(*sc, D);
  const double fh = (double)pow2f(-(ex.e_m + ex.e_a));
  __shared__ float part[32][16][4];
  __shared__ double vh[8][64];
  const int t = threadIdx.x;
  const int kb = blockIdx.x;
  const int g = blockIdx.y;
  const int hpg = H / G;
  const int R = hpg < 32 ? hpg : 32;   // heads per round
  const int P = 32 / R;                // row phases per head
  const int rows = n_chunks * GROUPS;
  const size_t run = (size_t)rows * 64;
  const int c4 = t & 15, rest = t >> 4;
  const int r = rest / P, ph = rest % P;
  // fp64 stage: thread t < 64 * min(R, 8) takes neuron n of head-in-round rr (more rounds of 8 if R > 8)
  const int n = t & 63;
  const int k = kb * 64 + n;
  double scale = 0.0;
  if (t < 64 * 8) scale = fh * fh * ((fo && k < I) ? (double)wdn[k] : 1.0) / (double)T;
  double total = 0.0;
  for (int h0 = g * hpg; h0 < (g + 1) * hpg; h0 += R) {
    const int nr = min(R, (g + 1) * hpg - h0);   // heads in this round
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < nr) {
      const float4* src = reinterpret_cast<const float4*>(partial + ((size_t)(h0 + r) * (I_pad / 64) + kb) * run) + c4;
#pragma unroll 8
      for (int row = ph; row < rows; row += P) {
        const float4 v = __ldg(src + (size_t)row * 16);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
    }
    part[rest][c4][0] = acc.x;
    part[rest][c4][1] = acc.y;
    part[rest][c4][2] = acc.z;
    part[rest][c4][3] = acc.w;
    __syncthreads();
    for (int rr0 = 0; rr0 < nr; rr0 += 8) {
      const int rr = rr0 + (t >> 6);
      if (t < 512 && rr < nr && (t >> 6) < 8) {
        double s = 0.0;
        for (int i = 0; i < P; ++i) s += part[rr * P + i][n >> 2][n & 3];
        const double v = s * scale;
        vh[t >> 6][n] = v;
        if (S_head_out && k < I) S_head_out[(size_t)(h0 + rr) * I + k] = (float)v;
      }
      __syncthreads();
      if (t < 64) {
        const int m = min(8, nr - rr0);
        for (int i = 0; i < m; ++i) total += vh[i][n];
      }
      __syncthreads();
    }
  }
  if (t < 64 && k < I) S_out[(size_t)g * I + k] = (float)total;
}

// S_head[h][k] = sum_t(...) / T (x ||w^d_k||^2 for FO); S_up[g][k] = sum_{h in g} S_head[h][k].
__global__ void finalize_up_kernel(const double* __restrict__ sh, const float* __restrict__ wdn, int fo, int T,
                                   int H, int G, int I, int I_pad, float* __restrict__ S_out,
                                   float* __restrict__ S_head_out) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  const int g = blockIdx.y;
  if (k >= I) return;
  const int hpg = H / G;
  const double scale = (fo ? (double)wdn[k] : 1.0) / (double)T;
  double s = 0.0;
  for (int h = g * hpg; h < (g + 1) * hpg; ++h) {
    const double v = sh[(size_t)h * I_pad + k] * scale;
    if (S_head_out) S_head_out[(size_t)h * I + k] = (float)v;
    s += v;
  }
  S_out[(size_t)g * I + k] = (float)s;
}

// ---------------------------------------------------------------- self-test of the bounded waits
// One thread waits on an mbarrier that nothing arrives at.  The wait must give
// up after limit_ns, latch the timeout status and return, leaving the context
// usable -- the path every pipeline wait of the tile kernel takes on a stall.
__global__ void wait_selftest_kernel(uint32_t* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status, limit_ns);
}

cudaError_t launch_wait_selftest(uint32_t* status, unsigned long long limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- leave-one-out score
// out = fp16 copy of n bf16 values (n % 8 == 0), 8 per thread.
__global__ void to_fp16_kernel(const uint16_t* __restrict__ in, __half* __restrict__ out, size_t n,
                               uint32_t* status) {
  pdl_enter();
  bool bad = false;
  for (size_t v = blockIdx.x * (size_t)blockDim.x + threadIdx.x; v < n / 8; v += (size_t)gridDim.x * blockDim.x) {
    uint4 q = *reinterpret_cast<const uint4*>(in + v * 8);
    const uint16_t* e = reinterpret_cast<const uint16_t*>(&q);
    __align__(16) __half o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = __float2half_rn(bf2f(e[i]));
    *reinterpret_cast<uint4*>(out + v * 8) = *reinterpret_cast<uint4*>(o);
  }
  if (bad) latch_status(status, kStatusRange);
}

// sigma[h][t] = 1 - rho with rho = r_t / rms(x_t - c_th), from the column groups of
// CC = sum_d (c/r)^2 and XD = sum_d x (c/r):  since mean_d x^2 = r^2 - eps,
//   rms(x - c)^2 / r^2 = 1 + q,  q = (CC - 2 XD / r) / D,
// and 1 - rho = 1 - 1/s = q / (s (s + 1)) with s = sqrt(1 + q), a form without
// cancellation when the head's write is small (rho near 1).  The leave-one-out
// change is then formed as p.w + sigma (g - p.w).  Padding tokens (t >= T) get
// sigma = 0; they carry no signal.
// The c_h pass contracted a16 (a/r 2^e_a) with Wo16 (Wo 2^e_o): its sums carry
// 2^(e_a + e_o) per factor of c/r, removed here.
__global__ void loo_rho_kernel(const float* __restrict__ cn, const float* __restrict__ inv_r, float* __restrict__ rho,
                               int T, int T_pad, int H, int D, int groups, const DevScales* __restrict__ sc) {
  pdl_enter();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  const int h = blockIdx.y;
  if (t >= T_pad) return;
  const ScaleExps ex = scale_exps(*sc, D);
  const float u = pow2f(-(ex.e_a + ex.e_o));
  float v = 0.0f;
  if (t < T) {
    const size_t plane = (size_t)H * T_pad, at = (size_t)h * T_pad + t;
    float cc = 0.f, xd = 0.f;   // column groups in order: [group][quantity][H][T_pad]
#pragma unroll 8
    for (int g = 0; g < groups; ++g) {
      cc += cn[(size_t)(2 * g) * plane + at];
      xd += cn[(size_t)(2 * g + 1) * plane + at];
    }
    cc = cc * u * u;
    xd = xd * u;
    const float q = (cc - 2.0f * xd * inv_r[t]) / (float)D;
    const float w = 1.0f + q;
    if (w > 1e-30f) {
      const float sq = sqrtf(w);
      v = q / (sq * (sq + 1.0f));
    } else {
      v = 1.0f - rsqrtf(1e-30f);   // x - c_h vanishes: rho at its clamp
    }
  }
  rho[(size_t)h * T_pad + t] = v;
}

// ---------------------------------------------------------------- down edge
// Wd16 [D][I_pad] and WdT16 [I_pad][D]: fp16 copies of Wd (zero padded).
__global__ void prep_wd_kernel(const uint16_t* __restrict__ Wd, __half* __restrict__ Wd16,
                               __half* __restrict__ WdT16, int D, int I, int I_pad, uint32_t* status) {
  pdl_enter();
  __shared__ float tile[32][33];
  const int d0 = blockIdx.y * 32, k0 = blockIdx.x * 32;
  bool bad = false;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int d = d0 + i, k = k0 + threadIdx.x;
    float v = 0.f;
    if (d < D && k < I) v = bf2f(Wd[(size_t)d * I + k]);
    tile[i][threadIdx.x] = v;
    if (d < D && k < I_pad) Wd16[(size_t)d * I_pad + k] = to_h(v, bad);
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int k = k0 + i, d = d0 + threadIdx.x;
    if (k < I_pad && d < D) WdT16[(size_t)k * D + d] = __float2half_rn(tile[threadIdx.x][i]);
  }
  if (bad) latch_status(status, kStatusRange);
}

// Wqkv16 [G][R_g][2][D]: rows of W^qkv_g (query rows of g's heads, then key, then
// value rows) times gamma', split into fp16 hi / lo.
__global__ void prep_qkv_kernel(const uint16_t* __restrict__ Wq, const uint16_t* __restrict__ Wk,
                                const uint16_t* __restrict__ Wv, const uint16_t* __restrict__ gamma_next,
                                __half* __restrict__ out, int G, int hpg, int dh, int D, uint32_t* status) {
  pdl_enter();
  const int Rg = (hpg + 2) * dh;
  const size_t total = (size_t)G * Rg * D;
  bool bad = false;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int d = (int)(e % D);
    const size_t rr = e / D;
    const int r = (int)(rr % Rg), g = (int)(rr / Rg);
    const uint16_t* src;
    if (r < hpg * dh) src = Wq + ((size_t)g * hpg * dh + r) * D;
    else if (r < (hpg + 1) * dh) src = Wk + ((size_t)g * dh + (r - hpg * dh)) * D;
    else src = Wv + ((size_t)g * dh + (r - (hpg + 1) * dh)) * D;
    const float v = bf2f(gamma_next[d]) * bf2f(src[d]);
    const __half hi = to_h(v, bad);
    out[(rr * 2 + 0) * D + d] = hi;
    out[(rr * 2 + 1) * D + d] = __float2half_rn(v - __half2float(hi));
  }
  if (bad) latch_status(status, kStatusRange);
}

// cpart[c][k] = sum over the tokens t of chunk c of alpha_tk^2 / r'_t^2, with
// 1/r'_t^2 = 1 / (sum_d x'_td^2 / D + eps) from the partial sums of ssx (one per
// column tile and column group of the x' pass).
// Block = one chunk of tokens x 1024 neurons (8 per thread, 16-byte loads of
// alpha); the chunk's token weights are formed once, in shared memory.
__global__ void down_token_weights_kernel(const __half* __restrict__ alpha16, const float* __restrict__ ssx,
                                          float* __restrict__ cpart, int T, int T_pad, int D, int I_pad,
                                          int chunk, float eps, int groups) {
  pdl_enter();
  extern __shared__ float w_tok[];   // [chunk]
  const int c = blockIdx.y;
  const int t0 = c * chunk, n = min(T, t0 + chunk) - t0;
  // two tokens per thread, their loads interleaved; the partial sums in their order
  for (int i = threadIdx.x; i < n; i += 2 * blockDim.x) {
    const int i2 = i + blockDim.x;
    const bool two = i2 < n;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
    for (int g = 0; g < groups; ++g) {
      const float* row = ssx + (size_t)g * T_pad + t0;
      s0 += row[i];
      if (two) s1 += row[i2];
    }
    w_tok[i] = 1.0f / (s0 / (float)D + eps);
    if (two) w_tok[i2] = 1.0f / (s1 / (float)D + eps);
  }
  __syncthreads();
  const int k0 = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (k0 >= I_pad) return;
  float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int i = 0; i < n; ++i) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(alpha16 + (size_t)(t0 + i) * I_pad + k0));
    const __half2* h = reinterpret_cast<const __half2*>(&q);
    const float w = w_tok[i];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(h[e]);
      s[2 * e] = fmaf(f.x * f.x, w, s[2 * e]);
      s[2 * e + 1] = fmaf(f.y * f.y, w, s[2 * e + 1]);
    }
  }
  float4* dst = reinterpret_cast<float4*>(cpart + (size_t)c * I_pad + k0);
  dst[0] = make_float4(s[0], s[1], s[2], s[3]);
  dst[1] = make_float4(s[4], s[5], s[6], s[7]);
}

// S_down[k][g] = (sum_c cpart[c][k] / T) * (bn[0][k][g] + bn[1][k][g])  (fp64 sums, fixed order)
// Block = 32 neurons x 8 warps; warp w sums chunks w, w + 8, ... and the eight
// partial sums are added in warp order.
__global__ void __launch_bounds__(256) finalize_down_kernel(const float* __restrict__ cpart,
                                                            const float* __restrict__ bnorm, int n_chunks,
                                                            int bhalves, int T, int I, int I_pad, int G,
                                                            float* __restrict__ S_out) {
  pdl_enter();
  __shared__ double part[8][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int k = blockIdx.x * 32 + lane;
  double cw = 0.0;
  if (k < I) {
#pragma unroll 8
    for (int i = w; i < n_chunks; i += 8) cw += (double)cpart[(size_t)i * I_pad + k];
  }
  part[w][lane] = cw;
  __syncthreads();
  if (w != 0 || k >= I) return;
  double c = 0.0;
#pragma unroll
  for (int q = 0; q < 8; ++q) c += part[q][lane];
  c /= (double)T;
  for (int g = 0; g < G; ++g) {
    double b = 0.0;
    for (int hf = 0; hf < bhalves; ++hf) b += (double)bnorm[((size_t)hf * I_pad + k) * G + g];
    S_out[(size_t)k * G + g] = (float)(c * b);
  }
}

// ---------------------------------------------------------------- fp32 path (CUDA cores)
__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

// inv_r[t]; n32 = gamma*x/r; a32 = a/r.  One block per token.
__global__ void f32_rows_kernel(const float* __restrict__ x, const float* __restrict__ a, const float* __restrict__ gamma,
                                float* __restrict__ n32, float* __restrict__ a32, float* __restrict__ inv_r, int D,
                                int HD, float eps) {
  __shared__ float red[32];
  const size_t t = blockIdx.x;
  float ss = 0.f;
  for (int d = threadIdx.x; d < D; d += blockDim.x) ss = fmaf(x[t * D + d], x[t * D + d], ss);
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];
    red[0] = s;
  }
  __syncthreads();
  const float ir = 1.0f / sqrtf(red[0] / (float)D + eps);
  if (threadIdx.x == 0 && inv_r) inv_r[t] = ir;
  for (int d = threadIdx.x; d < D; d += blockDim.x) n32[t * D + d] = gamma[d] * x[t * D + d] * ir;
  if (a32)
    for (int i = threadIdx.x; i < HD; i += blockDim.x) a32[t * HD + i] = a[t * HD + i] * ir;
}

// M32[2h + gu][k][j] = sum_d W[k][d] * gamma_d * Wo[d][h*dh + j]
__global__ void f32_fold_kernel(const float* __restrict__ Wg, const float* __restrict__ Wu, const float* __restrict__ gamma,
                                const float* __restrict__ Wo, float* __restrict__ M32, int H, int dh, int I, int D) {
  const size_t total = (size_t)2 * H * I * dh;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int j = (int)(e % dh);
    const int k = (int)((e / dh) % I);
    const int hg = (int)(e / ((size_t)dh * I));
    const int h = hg >> 1;
    const float* w = ((hg & 1) ? Wu : Wg) + (size_t)k * D;
    float s = 0.f;
    for (int d = 0; d < D; ++d) s = fmaf(w[d] * gamma[d], Wo[(size_t)d * H * dh + h * dh + j], s);
    M32[e] = s;
  }
}

// Per (t, k): g, u from n32; FO: ab[t][k] = (silu'(g) u, silu(g)); alpha32[t][k] = silu(g) u.
__global__ void f32_opoint_kernel(const float* __restrict__ n32, const float* __restrict__ Wg, const float* __restrict__ Wu,
                                  float2* __restrict__ ab, float* __restrict__ alpha32, int T, int D, int I) {
  const size_t total = (size_t)T * I;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int k = (int)(e % I);
    const size_t t = e / I;
    float g = 0.f, u = 0.f;
    for (int d = 0; d < D; ++d) {
      g = fmaf(n32[t * D + d], Wg[(size_t)k * D + d], g);
      u = fmaf(n32[t * D + d], Wu[(size_t)k * D + d], u);
    }
    const float s = sigmoidf_(g);
    if (ab) ab[e] = make_float2(s * (1.0f + g * (1.0f - s)) * u, g * s);
    if (alpha32) alpha32[e] = g * s * u;
  }
}

// partial[c][0][h][k] = sum_{t in chunk c} Delta^2 (FO) or pg^2 + pu^2 (ADD),
// with pg = sum_j a32[t][h*dh+j] M32[2h][k][j] (a32 already carries 1/r).
__global__ void f32_heads_kernel(const float* __restrict__ a32, const float* __restrict__ M32, const float2* __restrict__ ab,
                                 float* __restrict__ partial, int T, int H, int dh, int I, int chunk, int fo) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  const int h = blockIdx.y, c = blockIdx.z;
  if (k >= I) return;
  const float* mg = M32 + ((size_t)(2 * h) * I + k) * dh;
  const float* mu = M32 + ((size_t)(2 * h + 1) * I + k) * dh;
  float acc = 0.f;
  for (int t = c * chunk; t < min(T, (c + 1) * chunk); ++t) {
    const float* ar = a32 + (size_t)t * H * dh + h * dh;
    float pg = 0.f, pu = 0.f;
    for (int j = 0; j < dh; ++j) {
      pg = fmaf(ar[j], mg[j], pg);
      pu = fmaf(ar[j], mu[j], pu);
    }
    if (fo) {
      const float2 w = ab[(size_t)t * I + k];
      const float d = w.x * pg + w.y * pu;
      acc = fmaf(d, d, acc);
    } else {
      acc = fmaf(pg, pg, fmaf(pu, pu, acc));
    }
  }
  partial[((size_t)c * H + h) * I + k] = acc;
}

// ssx[t] = sum_d (x[t][d] + sum_k alpha[t][k] Wd[d][k])^2; the second half row stays 0.
__global__ void f32_xprime_kernel(const float* __restrict__ x, const float* __restrict__ alpha32, const float* __restrict__ Wd,
                                  float* __restrict__ ssx, int T, int T_pad, int D, int I) {
  __shared__ float red[32];
  const size_t t = blockIdx.x;
  float ss = 0.f;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float v = x[t * D + d];
    for (int k = 0; k < I; ++k) v = fmaf(alpha32[t * I + k], Wd[(size_t)d * I + k], v);
    ss = fmaf(v, v, ss);
  }
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];
    ssx[t] = s;
    ssx[(size_t)T_pad + t] = 0.f;
  }
}

// cpart[c][k] = sum_{t in chunk} alpha^2 / r'^2 for the fp32 path.
__global__ void f32_down_token_weights_kernel(const float* __restrict__ alpha32, const float* __restrict__ ssx,
                                              float* __restrict__ cpart, int T, int D, int I, int chunk, float eps) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  const int c = blockIdx.y;
  if (k >= I) return;
  float s = 0.f;
  for (int t = c * chunk; t < min(T, (c + 1) * chunk); ++t) {
    const float w = 1.0f / (ssx[t] / (float)D + eps);
    const float al = alpha32[(size_t)t * I + k];
    s = fmaf(al * al, w, s);
  }
  cpart[(size_t)c * I + k] = s;
}

// bnorm[0][k][g] = sum over W^qkv_g rows r of (sum_d Wrow[d] gamma'_d Wd[d][k])^2
__global__ void f32_qnorm_kernel(const float* __restrict__ Wq, const float* __restrict__ Wk, const float* __restrict__ Wv,
                                 const float* __restrict__ gamma_next, const float* __restrict__ Wd,
                                 float* __restrict__ bnorm, int hpg, int dh, int D, int I, int G) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  const int g = blockIdx.y;
  if (k >= I) return;
  const int Rg = (hpg + 2) * dh;
  float s = 0.f;
  for (int r = 0; r < Rg; ++r) {
    const float* row;
    if (r < hpg * dh) row = Wq + ((size_t)g * hpg * dh + r) * D;
    else if (r < (hpg + 1) * dh) row = Wk + ((size_t)g * dh + (r - hpg * dh)) * D;
    else row = Wv + ((size_t)g * dh + (r - (hpg + 1) * dh)) * D;
    float b = 0.f;
    for (int d = 0; d < D; ++d) b = fmaf(row[d] * gamma_next[d], Wd[(size_t)d * I + k], b);
    s = fmaf(b, b, s);
  }
  bnorm[(size_t)k * G + g] = s;
}

// ---------------------------------------------------------------- launchers
static inline int blocks_for(size_t n, int threads, int cap = 8192) {
  size_t b = (n + threads - 1) / threads;
  return (int)(b < (size_t)cap ? (b > 0 ? b : 1) : cap);
}

// At most 3 blocks of 8 warps per SM (a grid-stride loop over tokens): enough
// loads in flight to run near HBM speed, while leaving registers for the fold
// (one 320-thread CTA per SM), which runs concurrently on the side stream; at
// 4 blocks the two no longer fit one SM's register file together.  Measured on
// the Qwen3-shaped layer, the whole call: 8 blocks 2.406 ms, 4 blocks 2.388,
// 3 blocks 2.365, 2 blocks 2.374.  The
// kernel asks for the largest shared-memory carve-out although it uses none:
// an SM configured for a small carve-out could not take the fold's 214 KB CTA
// until it drained, which serialised the two.
cudaError_t launch_prep_tokens(const uint16_t* x, const uint16_t* a, const uint16_t* gamma, __half* n16, __half* a16,
                               float* inv_r, int T, int D, int HD, float eps, uint32_t* status, int sm_count,
                               DevScales* sc, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(prep_tokens_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  const int warps_per_block = 8;
  const int want = (T + warps_per_block - 1) / warps_per_block;
  const int cap = 3 * (sm_count > 0 ? sm_count : 1);
  if (cudaError_t e_ = launch_pdl(prep_tokens_kernel, want < cap ? want : cap, 32 * warps_per_block, 0, s, x, a,
                                  gamma, n16, a16, inv_r, T, D, HD, eps, status, sc); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

cudaError_t launch_restage_a(const uint16_t* a, const float* inv_r, __half* a16, int T, int HD, const DevScales* sc,
                             uint32_t* status, int sm_count, cudaStream_t s) {
  if (cudaError_t e_ = launch_pdl(restage_a_kernel, 4 * (sm_count > 0 ? sm_count : 1), 256, 0, s, a, inv_r, a16, T,
                                  HD, sc, status); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

cudaError_t launch_weight_stage(const uint16_t* Wg, const uint16_t* Wu, __half* W16, int I, int I_pad, int D,
                                const uint16_t* Wo, const uint16_t* gamma, __half* GWo16, int HD, DevScales* sc,
                                int sm_count, cudaStream_t s) {
  int g0 = (2 * I_pad + 7) / 8;                          // one warp per W16 row
  const int g1 = ((HD + 63) / 64) * ((D + 63) / 64);     // gamma*Wo^T tiles
  if (g0 < g1) g0 = g1;
  if (g0 > 8 * sm_count) g0 = 8 * (sm_count > 0 ? sm_count : 1);
  if (cudaError_t e_ = launch_pdl(weight_stage_kernel, dim3(g0, 2), 256, 0, s, Wg, Wu, W16, I, I_pad, D, Wo, gamma,
                                  GWo16, HD, sc); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

cudaError_t launch_weight_restage(const uint16_t* Wg, const uint16_t* Wu, __half* W16, int I, int I_pad, int D,
                                  const uint16_t* Wo, const uint16_t* gamma, __half* GWo16, __half* Wo16, int HD,
                                  DevScales* sc, uint32_t* status, int sm_count, cudaStream_t s) {
  if (cudaError_t e_ = launch_pdl(weight_restage_kernel, dim3(2 * (sm_count > 0 ? sm_count : 1), 3), 256, 0, s, Wg,
                                  Wu, W16, I, I_pad, D, Wo, gamma, GWo16, Wo16, HD, sc, status); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

cudaError_t launch_prep_gate_up(const uint16_t* Wg, const uint16_t* Wu, __half* W16, int I, int I_pad, int D,
                                DevScales* sc, cudaStream_t s) {
  if (cudaError_t e_ = launch_pdl(prep_gate_up_kernel, blocks_for((size_t)2 * I_pad, 8), 256, 0, s, Wg, Wu, W16, I,
                                  I_pad, D, sc); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

cudaError_t launch_wd_colnorm(const uint16_t* Wd, float* wdn, int D, int I, int I_pad, cudaStream_t s) {
  dim3 grid((I_pad + 31) / 32), block(32, 8);
  if (cudaError_t e_ = launch_pdl(wd_colnorm_kernel, grid, block, 0, s, Wd, wdn, D, I, I_pad); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

cudaError_t launch_wd_colnorm_f32(const float* Wd, float* wdn, int D, int I, cudaStream_t s) {
  dim3 grid((I + 31) / 32), block(32, 8);
  wd_colnorm_f32_kernel<<<grid, block, 0, s>>>(Wd, wdn, D, I);
  return cudaGetLastError();
}

cudaError_t launch_reduce_partials(const float* partial, double* out, int n_chunks, int halves, int H, int I_pad,
                                   cudaStream_t s) {
  if (I_pad % 128 == 0) {
    dim3 grid(I_pad / 128, H), block(32, 8);
    reduce_partials4_kernel<<<grid, block, 0, s>>>(partial, out, n_chunks, halves, H, I_pad);
  } else {
    dim3 grid((I_pad + 31) / 32, H), block(32, 8);
    reduce_partials_kernel<<<grid, block, 0, s>>>(partial, out, n_chunks, halves, H, I_pad);
  }
  return cudaGetLastError();
}

cudaError_t launch_reduce_finalize(const float* partial, const float* wdn, int fo, int n_chunks, int groups, int T,
                                   int H, int G, int I, int I_pad, float* S_out, float* S_head_out,
                                   const DevScales* sc, int D, cudaStream_t s) {
  dim3 grid(I_pad / 64, G), block(512);
  switch (groups) {
    case 1:
      if (cudaError_t e_ = launch_pdl(reduce_finalize_kernel<1>, grid, block, 0, s, partial, wdn, fo, n_chunks, T, H,
                                      G, I, I_pad, S_out, S_head_out, sc, D); e_ != cudaSuccess)
        return e_;
      break;
    case 2:
      if (cudaError_t e_ = launch_pdl(reduce_finalize_kernel<2>, grid, block, 0, s, partial, wdn, fo, n_chunks, T, H,
                                      G, I, I_pad, S_out, S_head_out, sc, D); e_ != cudaSuccess)
        return e_;
      break;
    case 4:
      if (cudaError_t e_ = launch_pdl(reduce_finalize_kernel<4>, grid, block, 0, s, partial, wdn, fo, n_chunks, T, H,
                                      G, I, I_pad, S_out, S_head_out, sc, D); e_ != cudaSuccess)
        return e_;
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_finalize_up(const double* sh, const float* wdn, int fo, int T, int H, int G, int I, int I_pad,
                               float* S_out, float* S_head_out, cudaStream_t s) {
  dim3 grid((I + 127) / 128, G);
  finalize_up_kernel<<<grid, 128, 0, s>>>(sh, wdn, fo, T, H, G, I, I_pad, S_out, S_head_out);
  return cudaGetLastError();
}

cudaError_t launch_to_fp16(const uint16_t* in, __half* out, size_t n, uint32_t* status, cudaStream_t s) {
  const size_t blocks = (n / 8 + 255) / 256;
  if (cudaError_t e_ = launch_pdl(to_fp16_kernel, (unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, s, in, out, n,
                                  status); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

cudaError_t launch_loo_rho(const float* cn, const float* inv_r, float* rho, int T, int T_pad, int H, int D,
                           int groups, const DevScales* sc, cudaStream_t s) {
  if (cudaError_t e_ = launch_pdl(loo_rho_kernel, dim3((T_pad + 255) / 256, H), 256, 0, s, cn, inv_r, rho, T, T_pad,
                                  H, D, groups, sc); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

cudaError_t launch_prep_wd(const uint16_t* Wd, __half* Wd16, __half* WdT16, int D, int I, int I_pad, uint32_t* status,
                           cudaStream_t s) {
  dim3 grid((I_pad + 31) / 32, (D + 31) / 32), block(32, 8);
  if (cudaError_t e_ = launch_pdl(prep_wd_kernel, grid, block, 0, s, Wd, Wd16, WdT16, D, I, I_pad, status); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

cudaError_t launch_prep_qkv(const uint16_t* Wq, const uint16_t* Wk, const uint16_t* Wv, const uint16_t* gamma_next,
                            __half* out, int G, int hpg, int dh, int D, uint32_t* status, cudaStream_t s) {
  if (cudaError_t e_ = launch_pdl(prep_qkv_kernel, blocks_for((size_t)G * (hpg + 2) * dh * D, 256), 256, 0, s, Wq, Wk,
                                  Wv, gamma_next, out, G, hpg, dh, D, status); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

cudaError_t launch_down_token_weights(const __half* alpha16, const float* ssx, float* cpart, int T, int T_pad, int D,
                                      int I_pad, int chunk, float eps, int groups, cudaStream_t s) {
  dim3 grid((I_pad / 8 + 127) / 128, (T + chunk - 1) / chunk);
  if (cudaError_t e_ = launch_pdl(down_token_weights_kernel, grid, 128, (size_t)chunk * sizeof(float), s, alpha16,
                                  ssx, cpart, T, T_pad, D, I_pad, chunk, eps, groups); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

cudaError_t launch_finalize_down(const float* cpart, const float* bnorm, int n_chunks, int bhalves, int T, int I,
                                 int I_pad, int G, float* S_out, cudaStream_t s) {
  if (cudaError_t e_ = launch_pdl(finalize_down_kernel, (I + 31) / 32, 256, 0, s, cpart, bnorm, n_chunks, bhalves, T,
                                  I, I_pad, G, S_out); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

cudaError_t launch_f32_up(const F32UpArgs& A, cudaStream_t s) {
  f32_rows_kernel<<<A.T, 128, 0, s>>>(A.x, A.a, A.gamma, A.n32, A.a32, nullptr, A.D, A.H * A.dh, A.eps);
  f32_fold_kernel<<<blocks_for((size_t)2 * A.H * A.I * A.dh, 128), 128, 0, s>>>(A.Wg, A.Wu, A.gamma, A.Wo, A.M32, A.H,
                                                                                 A.dh, A.I, A.D);
  if (A.fo)
    f32_opoint_kernel<<<blocks_for((size_t)A.T * A.I, 128), 128, 0, s>>>(A.n32, A.Wg, A.Wu, A.ab, nullptr, A.T, A.D,
                                                                          A.I);
  dim3 grid((A.I + 127) / 128, A.H, A.n_chunks);
  f32_heads_kernel<<<grid, 128, 0, s>>>(A.a32, A.M32, A.ab, A.partial, A.T, A.H, A.dh, A.I, A.chunk, A.fo);
  return cudaGetLastError();
}

cudaError_t launch_f32_down(const F32DownArgs& A, cudaStream_t s) {
  f32_rows_kernel<<<A.T, 128, 0, s>>>(A.x, nullptr, A.gamma, A.n32, nullptr, nullptr, A.D, 0, A.eps);
  f32_opoint_kernel<<<blocks_for((size_t)A.T * A.I, 128), 128, 0, s>>>(A.n32, A.Wg, A.Wu, nullptr, A.alpha32, A.T,
                                                                        A.D, A.I);
  f32_xprime_kernel<<<A.T, 128, 0, s>>>(A.x, A.alpha32, A.Wd, A.ssx, A.T, A.T, A.D, A.I);
  dim3 g1((A.I + 127) / 128, A.n_chunks);
  f32_down_token_weights_kernel<<<g1, 128, 0, s>>>(A.alpha32, A.ssx, A.cpart, A.T, A.D, A.I, A.chunk, A.eps);
  dim3 g2((A.I + 127) / 128, A.G);
  f32_qnorm_kernel<<<g2, 128, 0, s>>>(A.Wq, A.Wk, A.Wv, A.gamma_next, A.Wd, A.bnorm, A.H / A.G, A.dh, A.D, A.I, A.G);
  return cudaGetLastError();
}

}  // namespace aff
