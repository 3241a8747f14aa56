// tile_kernel.cu -- the persistent tcgen05 kernel behind every dense
// contraction of the affinity pass ("Affinity-Aware Sharding for Delayed
// Tensor Parallelism", §3 "Affinity scores").
//
// One CTA per SM (227 KB of shared memory, all 512 TMEM columns).  Warp
// roles:
//   warp 0       TMA producer: a ring of `stages` 48 KB stages, each holding
//                two 128 x 64 A tiles and one 128 x 64 B tile (fp16, 128 B
//                swizzle);
//   warp 1       MMA issuer (one thread): for every K slice of 16, two
//                tcgen05.mma (M=128, N=128) into a pair of fp32 accumulators
//                D1 = A1 B^T, D2 = A2 B^T in tensor memory; two such pairs
//                (buffers) alternate so the epilogue of one job overlaps the
//                MMAs of the next;
//   warps 2..9   epilogue: TMEM -> registers with tcgen05.ld; warp w reads
//                TMEM lanes 32*(w%4)..+31 (one row of A each) and half
//                (w-2)/4 of the 128 columns.
// Work is a fixed list of units, each a short list of jobs; CTAs take units
// round-robin.  Which CTA computes a unit never changes its result, and
// every unit writes its own partial sums, so the outputs do not depend on
// the grid size.
#include "sm103_primitives.cuh"
#include "tile_kernel.cuh"

#include <cuda_fp16.h>

namespace aff {

enum JobKind : int { kJobGateUp = 0, kJobHead = 1, kJobFold = 2, kJobXPrime = 3, kJobQNorm = 4 };

struct Job {
  int kind;
  int nkb;      // K blocks of 64
  int klen;     // valid K extent (for the last block's K-slice count)
  int head;     // head index (kJobHead)
  int part;     // fold: 0 = hi, 1 = lo half of gamma*Wo (selected per K block)
  int t0;       // first token (row of the B tile, or of A1 for x')
  int kt;       // neuron tile
  int nt;       // column / row tile
  int g;        // KV group (qnorm)
};

struct Unit {
  int njobs;
  int chunk;    // FO/ADD: token chunk index
  int kt;
  int tile0;    // FO/ADD/alpha: first token tile
  int base;     // x': first token; qnorm: first neuron
};

__device__ __forceinline__ Unit unit_info(const TileParams& p, int u) {
  Unit U{};
  switch (p.mode) {
    case kModeFold:
      U.kt = u % p.n_ktiles;
      U.njobs = 1;
      U.base = u / p.n_ktiles;  // column tile
      break;
    case kModeFO:
    case kModeADD:
    case kModeAlpha: {
      U.kt = u % p.n_ktiles;
      U.chunk = u / p.n_ktiles;
      U.tile0 = U.chunk * p.tiles_per_unit;
      int nt = min(p.tiles_per_unit, p.n_ttiles - U.tile0);
      int per = p.mode == kModeFO ? 1 + p.H : (p.mode == kModeADD ? p.H : 1);
      U.njobs = nt * per;
      break;
    }
    case kModeXPrime:
      U.base = u * 2 * kBlockM;
      U.njobs = p.n_ntiles;
      break;
    case kModeQNorm:
      U.base = u * 2 * kBlockM;
      U.njobs = p.G * p.n_ntiles;
      break;
  }
  return U;
}

__device__ __forceinline__ Job job_info(const TileParams& p, const Unit& U, int j) {
  Job J{};
  J.kt = U.kt;
  switch (p.mode) {
    case kModeFold:
      J.kind = kJobFold;
      J.nkb = 2 * p.nkb_D;
      J.klen = p.D;
      J.nt = U.base;
      break;
    case kModeFO: {
      int per = 1 + p.H;
      int tile = U.tile0 + j / per, r = j % per;
      J.t0 = tile * kBlockN;
      if (r == 0) {
        J.kind = kJobGateUp; J.nkb = p.nkb_D; J.klen = p.D;
      } else {
        J.kind = kJobHead; J.head = r - 1; J.nkb = p.nkb_dh; J.klen = p.dh;
      }
      break;
    }
    case kModeADD: {
      int tile = U.tile0 + j / p.H;
      J.t0 = tile * kBlockN;
      J.kind = kJobHead; J.head = j % p.H; J.nkb = p.nkb_dh; J.klen = p.dh;
      break;
    }
    case kModeAlpha:
      J.t0 = (U.tile0 + j) * kBlockN;
      J.kind = kJobGateUp; J.nkb = p.nkb_D; J.klen = p.D;
      break;
    case kModeXPrime:
      J.kind = kJobXPrime; J.nkb = p.nkb_I; J.klen = p.I_pad;
      J.t0 = U.base; J.nt = j;
      break;
    case kModeQNorm:
      J.kind = kJobQNorm; J.nkb = 2 * p.nkb_D; J.klen = p.D;
      J.g = j / p.n_ntiles; J.nt = j % p.n_ntiles;
      break;
  }
  return J;
}

// Number of 16-wide K slices in K block kb of a job.
__device__ __forceinline__ int kslices(const Job& J, int kb, int nkb_D) {
  int k_in = (J.kind == kJobFold || J.kind == kJobQNorm) ? (kb % nkb_D) : kb;
  int rem = J.klen - k_in * kBlockK;
  int n = (rem + 15) >> 4;
  return n < 4 ? n : 4;
}

struct Smem {
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tfull;
  uint64_t* tempty;
  uint64_t* drain;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  float* sacc;
  uint8_t* stage0;
};

__device__ __forceinline__ float h_lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu))); }
__device__ __forceinline__ float h_hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    affinity_tile_kernel(const __grid_constant__ CUtensorMap map0, const __grid_constant__ CUtensorMap map1,
                         const __grid_constant__ CUtensorMap map2, const __grid_constant__ CUtensorMap map3,
                         const TileParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);

  const int S = p.stages;
  Smem sm;
  sm.stage0 = base;
  uint8_t* cur = base + (size_t)S * kStageBytes;
  sm.sacc = reinterpret_cast<float*>(cur);
  int sacc_floats = (MODE == kModeFO || MODE == kModeADD) ? 2 * p.H * kBlockM : 0;
  cur += (size_t)sacc_floats * 4;
  sm.full = reinterpret_cast<uint64_t*>(cur);
  sm.empty = sm.full + S;
  sm.tfull = sm.empty + S;
  sm.tempty = sm.tfull + 2;
  sm.drain = sm.tempty + 2;
  sm.tmem_slot = reinterpret_cast<uint32_t*>(sm.drain + 1);
  sm.abort_flag = reinterpret_cast<volatile int*>(sm.tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.tfull[b], 1);
      mbar_init(&sm.tempty[b], kEpiWarps);
    }
    mbar_init(sm.drain, 1);
    *sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map0);
    prefetch_tmap(&map1);
    prefetch_tmap(&map2);
    prefetch_tmap(&map3);
  }
  if (warp == 1) {
    tmem_alloc(sm.tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 2) {
    for (int i = threadIdx.x - 64; i < sacc_floats; i += kEpiWarps * 32) sm.sacc[i] = 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
        Unit U = unit_info(p, u);
        for (int j = 0; ok && j < U.njobs; ++j) {
          Job J = job_info(p, U, j);
          for (int kb = 0; kb < J.nkb; ++kb, ++it) {
            const int s = it % S;
            const uint32_t k = (uint32_t)(it / S);
            if (!mbar_wait(&sm.empty[s], (k & 1u) ^ 1u, sm.abort_flag, p.status)) { ok = false; break; }
            uint8_t* st = sm.stage0 + (size_t)s * kStageBytes;
            uint64_t* fb = &sm.full[s];
            mbar_arrive_expect_tx(fb, kStageBytes);
            const int kx = kb * kBlockK;
            switch (J.kind) {
              case kJobGateUp:   // A = W16 gate / up rows, B = n16 token rows
                tma_load_2d(st, &map0, fb, kx, J.kt * kBlockM);
                tma_load_2d(st + kTileBytes, &map0, fb, kx, p.I_pad + J.kt * kBlockM);
                tma_load_2d(st + 2 * kTileBytes, &map1, fb, kx, J.t0);
                break;
              case kJobHead:     // A = M16 (gate, up) of head h, B = a16 head h
                tma_load_3d(st, &map2, fb, kx, J.kt * kBlockM, 2 * J.head);
                tma_load_3d(st + kTileBytes, &map2, fb, kx, J.kt * kBlockM, 2 * J.head + 1);
                tma_load_3d(st + 2 * kTileBytes, &map3, fb, kx, J.head, J.t0);
                break;
              case kJobFold: {   // A = W16 rows, B = gamma*Wo^T (hi or lo part)
                const int part = kb / p.nkb_D, kxp = (kb % p.nkb_D) * kBlockK;
                tma_load_2d(st, &map0, fb, kxp, J.kt * kBlockM);
                tma_load_2d(st + kTileBytes, &map0, fb, kxp, p.I_pad + J.kt * kBlockM);
                tma_load_3d(st + 2 * kTileBytes, &map1, fb, kxp, part, J.nt * kBlockN);
                break;
              }
              case kJobXPrime:   // A = alpha16 token rows (two tiles), B = Wd16 rows d
                tma_load_2d(st, &map0, fb, kx, J.t0);
                tma_load_2d(st + kTileBytes, &map0, fb, kx, J.t0 + kBlockM);
                tma_load_2d(st + 2 * kTileBytes, &map1, fb, kx, J.nt * kBlockN);
                break;
              case kJobQNorm: {  // A = Wd^T neuron rows (two tiles), B = group g's gamma'-scaled q/k/v rows (hi | lo)
                const int part = kb / p.nkb_D, kxp = (kb % p.nkb_D) * kBlockK;
                tma_load_2d(st, &map0, fb, kxp, U.base);
                tma_load_2d(st + kTileBytes, &map0, fb, kxp, U.base + kBlockM);
                tma_load_4d(st + 2 * kTileBytes, &map1, fb, kxp, part, J.nt * kBlockN, J.g);
                break;
              }
            }
          }
        }
      }
      if (!ok) {
        // Let every copy already issued land before shared memory is released.
        const int n = it < S ? it : S;
        for (int i = 1; i <= n; ++i) {
          const int q = it - i;
          volatile int dummy = 0;
          mbar_wait(&sm.full[q % S], (uint32_t)((q / S) & 1), &dummy, p.status, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kBlockM, kBlockN, 0);
      int it = 0, jc = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
        Unit U = unit_info(p, u);
        for (int j = 0; ok && j < U.njobs; ++j, ++jc) {
          Job J = job_info(p, U, j);
          const int b = jc & 1;
          if (!mbar_wait(&sm.tempty[b], (uint32_t)(((jc >> 1) & 1) ^ 1), sm.abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d1 = tmem + (uint32_t)(b * 2 * kBlockN);
          const uint32_t d2 = d1 + kBlockN;
          for (int kb = 0; kb < J.nkb; ++kb, ++it) {
            const int s = it % S;
            const uint32_t k = (uint32_t)(it / S);
            if (!mbar_wait(&sm.full[s], k & 1u, sm.abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t st = smem_u32(sm.stage0 + (size_t)s * kStageBytes);
            const uint64_t da1 = smem_desc_k_sw128(st);
            const uint64_t da2 = smem_desc_k_sw128(st + kTileBytes);
            const uint64_t db = smem_desc_k_sw128(st + 2 * kTileBytes);
            const int nks = kslices(J, kb, p.nkb_D);
            for (int ks = 0; ks < nks; ++ks) {
              const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
              mma_f16_ss(d1, da1 + 2 * ks, db + 2 * ks, idesc, acc);
              mma_f16_ss(d2, da2 + 2 * ks, db + 2 * ks, idesc, acc);
            }
            mma_commit(&sm.empty[s]);
          }
          if (!ok) break;
          mma_commit(&sm.tfull[b]);
        }
      }
      if (!ok) {
        mma_commit(sm.drain);
        volatile int dummy = 0;
        mbar_wait(sm.drain, 0, &dummy, p.status, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quarter this warp may read
    const int hf = (warp - 2) >> 2;    // which 64-column half of the tile
    const int row = q * 32 + lane;     // row of the A tile = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t abA[32], abB[32];         // FO: fp16 pairs of silu'(g)u and silu(g), 64 tokens
#pragma unroll
    for (int i = 0; i < 32; ++i) { abA[i] = 0u; abB[i] = 0u; }
    float ss1 = 0.f, ss2 = 0.f;        // x' / qnorm running sums
    int jc = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
      Unit U = unit_info(p, u);
      for (int j = 0; j < U.njobs; ++j, ++jc) {
        Job J = job_info(p, U, j);
        const int b = jc & 1;
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait(&sm.tfull[b], (uint32_t)((jc >> 1) & 1), sm.abort_flag, p.status) ? 1 : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) { ok = false; break; }
        tc_fence_after();
        const uint32_t c1 = tl + (uint32_t)(b * 2 * kBlockN + hf * 64);
        const uint32_t c2 = c1 + kBlockN;

        if constexpr (MODE == kModeFO || MODE == kModeAlpha) {
          if (J.kind == kJobGateUp) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t gr[16], ur[16];
              tmem_ld16(c1 + c * 16, gr);
              tmem_ld16(c2 + c * 16, ur);
              tmem_ld_wait();
              if (c == 3) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.tempty[b]);
              }
#pragma unroll
              for (int i = 0; i < 16; i += 2) {
                float gA[2], gB[2], al[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const float g = __uint_as_float(gr[i + e]);
                  const float uu = __uint_as_float(ur[i + e]);
                  const float sg = __frcp_rn(1.0f + __expf(-g));        // sigmoid(g)
                  const float si = g * sg;                              // silu(g)
                  gA[e] = sg * fmaf(g, 1.0f - sg, 1.0f) * uu;           // silu'(g) u
                  gB[e] = si;
                  al[e] = si * uu;                                      // alpha = silu(g) u
                }
                if constexpr (MODE == kModeFO) {
                  abA[c * 8 + i / 2] = pack_h2(gA[0], gA[1]);
                  abB[c * 8 + i / 2] = pack_h2(gB[0], gB[1]);
                } else {
                  const int t = J.t0 + hf * 64 + c * 16 + i;
                  const int kk = J.kt * kBlockM + row;
                  p.alpha16[(size_t)t * p.I_pad + kk] = __float2half_rn(al[0]);
                  p.alpha16[(size_t)(t + 1) * p.I_pad + kk] = __float2half_rn(al[1]);
                }
              }
            }
            continue;
          }
        }
        if constexpr (MODE == kModeFO || MODE == kModeADD) {
          // kJobHead: per token Delta = A' pg + B' pu (FO) or pg^2 + pu^2 (ADD), summed over tokens
          uint64_t acc = pk(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pg[16], pu[16];
            tmem_ld16(c1 + c * 16, pg);
            tmem_ld16(c2 + c * 16, pu);
            tmem_ld_wait();
            if (c == 3) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.tempty[b]);
            }
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const uint64_t vg = pk_u(pg[i], pg[i + 1]);
              const uint64_t vu = pk_u(pu[i], pu[i + 1]);
              if constexpr (MODE == kModeFO) {
                const uint32_t wa = abA[c * 8 + i / 2], wb = abB[c * 8 + i / 2];
                const uint64_t va = pk(h_lo(wa), h_hi(wa));
                const uint64_t vb = pk(h_lo(wb), h_hi(wb));
                uint64_t d = mul2(va, vg);
                d = fma2(vb, vu, d);
                acc = fma2(d, d, acc);
              } else {
                acc = fma2(vg, vg, acc);
                acc = fma2(vu, vu, acc);
              }
            }
          }
          const float2 s2 = unpk(acc);
          sm.sacc[(hf * p.H + J.head) * kBlockM + row] += s2.x + s2.y;
        }
        if constexpr (MODE == kModeFold) {
          // D1 = Mg[k][n], D2 = Mu[k][n] for neuron k = kt*128 + row, columns n = nt*128 + hf*64 + ...
          const int kk = J.kt * kBlockM + row;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t mg[16], mu[16];
            tmem_ld16(c1 + c * 16, mg);
            tmem_ld16(c2 + c * 16, mu);
            tmem_ld_wait();
            if (c == 3) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.tempty[b]);
            }
#pragma unroll
            for (int i = 0; i < 16; i += 8) {
              const int n = J.nt * kBlockN + hf * 64 + c * 16 + i;
              if (n < p.H * p.dh) {
                const int h = n / p.dh, jj = n % p.dh;
                uint4 vg, vu;
                vg.x = pack_h2(__uint_as_float(mg[i + 0]), __uint_as_float(mg[i + 1]));
                vg.y = pack_h2(__uint_as_float(mg[i + 2]), __uint_as_float(mg[i + 3]));
                vg.z = pack_h2(__uint_as_float(mg[i + 4]), __uint_as_float(mg[i + 5]));
                vg.w = pack_h2(__uint_as_float(mg[i + 6]), __uint_as_float(mg[i + 7]));
                vu.x = pack_h2(__uint_as_float(mu[i + 0]), __uint_as_float(mu[i + 1]));
                vu.y = pack_h2(__uint_as_float(mu[i + 2]), __uint_as_float(mu[i + 3]));
                vu.z = pack_h2(__uint_as_float(mu[i + 4]), __uint_as_float(mu[i + 5]));
                vu.w = pack_h2(__uint_as_float(mu[i + 6]), __uint_as_float(mu[i + 7]));
                *reinterpret_cast<uint4*>(p.M16 + ((size_t)(2 * h) * p.I_pad + kk) * p.dh + jj) = vg;
                *reinterpret_cast<uint4*>(p.M16 + ((size_t)(2 * h + 1) * p.I_pad + kk) * p.dh + jj) = vu;
              }
            }
          }
        }
        if constexpr (MODE == kModeXPrime) {
          // D1 = (alpha Wd^T)[t1][d], D2 = ...[t2][d]; x' = x + D; accumulate x'^2 over d
          const int t1 = J.t0 + row, t2 = J.t0 + kBlockM + row;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t v1[16], v2[16];
            tmem_ld16(c1 + c * 16, v1);
            tmem_ld16(c2 + c * 16, v2);
            tmem_ld_wait();
            if (c == 3) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.tempty[b]);
            }
            const int d0 = J.nt * kBlockN + hf * 64 + c * 16;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int d = d0 + i;
              if (d < p.D) {
                if (t1 < p.T) {
                  const float xv = __uint_as_float((uint32_t)p.x_bf16[(size_t)t1 * p.D + d] << 16);
                  const float v = xv + __uint_as_float(v1[i]);
                  ss1 = fmaf(v, v, ss1);
                }
                if (t2 < p.T) {
                  const float xv = __uint_as_float((uint32_t)p.x_bf16[(size_t)t2 * p.D + d] << 16);
                  const float v = xv + __uint_as_float(v2[i]);
                  ss2 = fmaf(v, v, ss2);
                }
              }
            }
          }
        }
        if constexpr (MODE == kModeQNorm) {
          // D1 = Q[k1][r], D2 = Q[k2][r] for the rows r of group J.g; sum Q^2 over the group's rows
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t v1[16], v2[16];
            tmem_ld16(c1 + c * 16, v1);
            tmem_ld16(c2 + c * 16, v2);
            tmem_ld_wait();
            if (c == 3) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.tempty[b]);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float a1 = __uint_as_float(v1[i]), a2 = __uint_as_float(v2[i]);
              ss1 = fmaf(a1, a1, ss1);
              ss2 = fmaf(a2, a2, ss2);
            }
          }
          if (J.nt == p.n_ntiles - 1) {
            // rows past the group's end were zero-filled, so the sum is the group's ||b_gk||^2 half
            const int k1 = U.base + row, k2 = U.base + kBlockM + row;
            if (k1 < p.I_pad) p.bnorm[((size_t)hf * p.I_pad + k1) * p.G + J.g] = ss1;
            if (k2 < p.I_pad) p.bnorm[((size_t)hf * p.I_pad + k2) * p.G + J.g] = ss2;
            ss1 = 0.f;
            ss2 = 0.f;
          }
        }
      }
      if (!ok) break;
      // ---- end of unit
      if constexpr (MODE == kModeFO || MODE == kModeADD) {
        float* dst = p.partial + ((size_t)(U.chunk * 2 + hf) * p.H) * p.I_pad + U.kt * kBlockM + row;
        for (int h = 0; h < p.H; ++h) {
          float* sp = &sm.sacc[(hf * p.H + h) * kBlockM + row];
          dst[(size_t)h * p.I_pad] = *sp;
          *sp = 0.f;
        }
      }
      if constexpr (MODE == kModeXPrime) {
        const int t1 = U.base + row, t2 = U.base + kBlockM + row;
        if (t1 < p.T_pad) p.partial[(size_t)hf * p.T_pad + t1] = ss1;
        if (t2 < p.T_pad) p.partial[(size_t)hf * p.T_pad + t2] = ss2;
        ss1 = 0.f;
        ss2 = 0.f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

size_t tile_smem_bytes(int mode, int stages, int H) {
  size_t sacc = (mode == kModeFO || mode == kModeADD) ? (size_t)2 * H * kBlockM * 4 : 0;
  return 1024 + (size_t)stages * kStageBytes + sacc + (size_t)(2 * stages + 5) * 8 + 8;
}

template <int MODE>
static cudaError_t launch_mode(const CUtensorMap* maps, const TileParams& p, int grid, cudaStream_t stream) {
  const size_t smem = tile_smem_bytes(MODE, p.stages, p.H);
  cudaError_t e = cudaFuncSetAttribute(affinity_tile_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  affinity_tile_kernel<MODE><<<grid, kThreads, smem, stream>>>(maps[0], maps[1], maps[2], maps[3], p);
  return cudaGetLastError();
}

cudaError_t launch_tile_kernel(const CUtensorMap* maps, const TileParams& p, int grid, cudaStream_t stream) {
  switch (p.mode) {
    case kModeFold: return launch_mode<kModeFold>(maps, p, grid, stream);
    case kModeFO: return launch_mode<kModeFO>(maps, p, grid, stream);
    case kModeADD: return launch_mode<kModeADD>(maps, p, grid, stream);
    case kModeAlpha: return launch_mode<kModeAlpha>(maps, p, grid, stream);
    case kModeXPrime: return launch_mode<kModeXPrime>(maps, p, grid, stream);
    case kModeQNorm: return launch_mode<kModeQNorm>(maps, p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace aff
