// moment_kernel.cu -- the ADD score through each head's second moment (see
// moment_kernel.cuh): the per-token rms, the tcgen05 Gram pass that reads the
// bf16 head outputs itself, its deterministic reduction, and the tcgen05
// quadratic-form pass over the folded rows.  Paper: "Affinity-Aware Sharding
// for Delayed Tensor Parallelism", §3 "Affinity scores" (the ADD score).
#include "moment_kernel.cuh"
#include "launch.cuh"
#include "scales.cuh"
#include "sm103_primitives.cuh"

namespace aff {

namespace {

__device__ __forceinline__ float bf2f_m(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

}  // namespace

// ---------------------------------------------------------------- token rms
// inv_r[t] = 1 / sqrt(mean_d x_t,d^2 + eps) for t < T, 0 for T <= t < n_pad; one
// warp per token, two tokens' loads in flight together (per token the same sum
// order as the token-major staging of the other passes).
__global__ void __launch_bounds__(256) inv_r_kernel(const uint16_t* __restrict__ x, float* __restrict__ inv_r, int T,
                                                    int n_pad, int D, float eps) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int n_warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * 2; t < n_pad; t += 2 * n_warps) {
    const bool v0 = t < T, v1 = t + 1 < T;
    const uint4* x0 = reinterpret_cast<const uint4*>(x + (size_t)(v0 ? t : 0) * D);
    const uint4* x1 = reinterpret_cast<const uint4*>(x + (size_t)(v1 ? t + 1 : 0) * D);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll 4
    for (int v = lane; v < D / 8; v += 32) {
      const uint4 p0 = __ldg(x0 + v), p1 = __ldg(x1 + v);
      const uint16_t* e0 = reinterpret_cast<const uint16_t*>(&p0);
      const uint16_t* e1 = reinterpret_cast<const uint16_t*>(&p1);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float f0 = bf2f_m(e0[i]), f1 = bf2f_m(e1[i]);
        s0 = fmaf(f0, f0, s0);
        s1 = fmaf(f1, f1, s1);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, o);
      s1 += __shfl_xor_sync(0xffffffffu, s1, o);
    }
    if (lane == 0) {
      inv_r[t] = v0 ? rsqrtf(s0 / (float)D + eps) : 0.f;
      if (t + 1 < n_pad) inv_r[t + 1] = v1 ? rsqrtf(s1 / (float)D + eps) : 0.f;
    }
  }
}

// ---------------------------------------------------------------- Gram reduction
// Block = (head h, 2 rows n).  s_h = the sum over chunks of each chunk's
// largest diagonal entry (in chunk order; every block computes the same value),
// an upper bound on max_i C_h[i][i], so |C_h[n][i]| <= sqrt(C_ii C_nn) <= s_h.
// Each entry is summed in chunk order and C_h / s_h is split into an fp16 high
// part and the fp16 rounding of the remainder.
//
// The Gram pass staged a/r in fp16 unscaled.  If any head's s_h is not finite
// (an operand overflowed fp16) or every head's s_h is below T 2^-16 (a/r so
// small that fp16 subnormals would cost precision), the matrices are instead
// recomputed with a power-of-two scale by moment_fallback_kernel: this kernel
// then records that decision, adds its share of max |a/r| over all tokens to
// sc->amax2, and writes nothing else.
constexpr int kReduceRows = 2;   // one entry of C_h per thread

__global__ void __launch_bounds__(256) gram_reduce_kernel(const float* __restrict__ gram,
                                                          const float* __restrict__ cmax, __half* __restrict__ CC,
                                                          float* __restrict__ scale, int n_chunks, int H, int dh,
                                                          uint32_t* status, const uint16_t* __restrict__ a,
                                                          const float* __restrict__ inv_r, int T, DevScales* sc) {
  pdl_enter();
  __shared__ float s_sh;
  __shared__ int redo_s;
  __shared__ uint32_t top_s;
  const int h = blockIdx.x, y = blockIdx.y;
  const size_t cstride = (size_t)H * 128 * 128;
  const float* g0 = gram + (size_t)h * 128 * 128;
  if (threadIdx.x == 0) top_s = 0u;
  __syncthreads();
  // every head's s_h (a thread per head, chunks in order; the loads eight at a time ahead
  // of the sum): any not finite, and the largest.  The thread of head h keeps its sum.
  bool nonfinite = false;
  float top = 0.f;
  for (int hh = threadIdx.x; hh < H; hh += 256) {
    float m = 0.f;
    int c = 0;
    for (; c + 8 <= n_chunks; c += 8) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = cmax[(size_t)(c + j) * H + hh];
#pragma unroll
      for (int j = 0; j < 8; ++j) m += v[j];
    }
    for (; c < n_chunks; ++c) m += cmax[(size_t)c * H + hh];
    if (hh == h) s_sh = m;
    if (isfinite(m)) top = fmaxf(top, m);
    else nonfinite = true;
  }
  atomicMax(&top_s, __float_as_uint(top));   // top >= 0: bit patterns order like the values
  const int any_nonfinite = __syncthreads_or(nonfinite ? 1 : 0);
  if (threadIdx.x == 0) {
    redo_s = (any_nonfinite || __uint_as_float(top_s) < (float)T * (1.0f / 65536.0f)) ? 1 : 0;
    float m = s_sh;
    if (!(m > 0.f) || !isfinite(m)) m = 1.f;
    s_sh = m;
    if (h == 0 && y == 0) sc->redo = (uint32_t)redo_s;
    if (!redo_s && y == 0) scale[h] = m;
  }
  __syncthreads();
  if (redo_s) {
    // this block's share of max |a/r| over every token (HD = H dh columns)
    const int HD = H * dh;
    const size_t n = (size_t)T * HD;
    const size_t nb = (size_t)gridDim.x * gridDim.y, b = (size_t)y * gridDim.x + h;
    uint32_t am = 0u;
    for (size_t e = b * 256 + threadIdx.x; e < n; e += nb * 256) {
      const float v = bf2f_m(a[e]) * inv_r[e / HD];
      am = max(am, __float_as_uint(fabsf(v)));
    }
    am = __reduce_max_sync(0xffffffffu, am);
    if ((threadIdx.x & 31) == 0 && am) atomicMax(&sc->amax2, am);
    return;
  }
  const float s = s_sh;
  for (int e = threadIdx.x; e < kReduceRows * 128; e += 256) {
    const int n = y * kReduceRows + (e >> 7), i = e & 127;
    float v = 0.f;
    if (n < dh && i < dh) {
      const float* src = g0 + (size_t)n * 128 + i;
#pragma unroll 8
      for (int c = 0; c < n_chunks; ++c) v += __ldg(src + c * cstride);
      v = v / s;
    }
    const __half hi = __float2half_rn(v);
    const __half lo = __float2half_rn(v - __half2float(hi));
    CC[((size_t)h * 128 + n) * 128 + i] = hi;
    CC[((size_t)(H + h) * 128 + n) * 128 + i] = lo;
  }
}

// The Gram matrices recomputed with a scale, when gram_reduce_kernel asked for it
// (otherwise every block returns at once).  One block per head: a~ = a/r 2^e,
// e from sc->amax2 (a non-finite maximum latches AFF_ERR_RANGE), tokens in order
// through shared memory in tiles of 32, C_h in fp32 on the CUDA cores; then
// s = max_i C_h[i][i], CC = [hi; lo] of C_h / s and scale[h] = s 2^-2e, the
// same outputs as gram_reduce_kernel.  Slow (about a millisecond per head) but
// only taken for inputs outside fp16's range.
constexpr int kFbTile = 32;

__global__ void __launch_bounds__(1024) moment_fallback_kernel(const uint16_t* __restrict__ a,
                                                              const float* __restrict__ inv_r, int T, int H, int dh,
                                                              __half* __restrict__ CC, float* __restrict__ scale,
                                                              const DevScales* __restrict__ sc, uint32_t* status) {
  pdl_enter();
  if (sc->redo == 0u) return;
  const float am = bits_f(sc->amax2);
  if (!(am <= 3.4e38f)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) latch_status(status, kStatusRange);
    return;
  }
  const int e = scale_exp_norm(am);
  const float f = pow2f(e);
  const int h = blockIdx.x, HD = H * dh;
  __shared__ float tile[kFbTile][128];
  __shared__ float dmax_s;
  const int i = threadIdx.x >> 3, j0 = (threadIdx.x & 7) * 16;   // row i, columns j0 .. j0+15
  float acc[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) acc[q] = 0.f;
  for (int t0 = 0; t0 < T; t0 += kFbTile) {
    __syncthreads();
    for (int v = threadIdx.x; v < kFbTile * 128; v += 1024) {
      const int tt = v >> 7, c = v & 127, t = t0 + tt;
      tile[tt][c] = (t < T && c < dh) ? bf2f_m(a[(size_t)t * HD + (size_t)h * dh + c]) * inv_r[t] * f : 0.f;
    }
    __syncthreads();
    if (i < dh) {
#pragma unroll 4
      for (int tt = 0; tt < kFbTile; ++tt) {
        const float ai = tile[tt][i];
#pragma unroll
        for (int q = 0; q < 16; ++q) acc[q] = fmaf(ai, tile[tt][j0 + q], acc[q]);
      }
    }
  }
  if (threadIdx.x == 0) dmax_s = 0.f;
  __syncthreads();
  if (i < dh && i >= j0 && i < j0 + 16) atomicMax(reinterpret_cast<unsigned int*>(&dmax_s), __float_as_uint(acc[i - j0]));
  __syncthreads();
  float s = dmax_s;
  if (!(s > 0.f) || !isfinite(s)) s = 1.f;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int j = j0 + q;
    const float v = (i < dh && j < dh) ? acc[q] / s : 0.f;
    const __half hi = __float2half_rn(v);
    const __half lo = __float2half_rn(v - __half2float(hi));
    CC[((size_t)h * 128 + i) * 128 + j] = hi;
    CC[((size_t)(H + h) * 128 + i) * 128 + j] = lo;
  }
  if (threadIdx.x == 0) scale[h] = s * pow2f(-e) * pow2f(-e);
}

// ---------------------------------------------------------------- finishing
// S_head[h][k] = out[h][k] / T; S_up[g][k] = the sum of S_head over g's heads in
// head order (fp64).  One thread per (group, neuron).
// The folded rows were staged times 2^e_m, so the quadratic forms carry 2^2e_m.
__global__ void __launch_bounds__(256) moment_finalize_kernel(const float* __restrict__ out, int T, int H, int G,
                                                              int I, int I_pad, float* __restrict__ S_out,
                                                              float* __restrict__ S_head_out,
                                                              const DevScales* __restrict__ sc, int D) {
  pdl_enter();
  const int k = blockIdx.x * 256 + threadIdx.x, g = blockIdx.y;
  if (k >= I) return;
  const int hpg = H / G;
  const double fm = (double)pow2f(-scale_exps(*sc, D).e_m);
  const double invT = fm * fm / (double)T;
  double total = 0.0;
  for (int h = g * hpg; h < (g + 1) * hpg; ++h) {
    const double v = (double)out[(size_t)h * I_pad + k] * invT;
    if (S_head_out) S_head_out[(size_t)h * I + k] = (float)v;
    total += v;
  }
  S_out[(size_t)g * I + k] = (float)total;
}

// ---------------------------------------------------------------- tcgen05 passes
// One unit per CTA: warp 0 issues the TMA copies, warp 1 the MMAs (one
// 128 x 128 fp32 accumulator in TMEM), warps 2..5 convert (Gram) and read the
// accumulator back.
//   Gram: unit (head h, token chunk c).  Per block of 64 tokens the TMA copies the
//         head's d_head bf16 columns of a ([64][d_head], unswizzled) and the block's
//         64 values of 1/r into a raw stage; the converter warps write a~ = fp16(a/r)
//         transposed into a 128-row K-major operand tile (128 B swizzle, rows past
//         d_head zeroed once), the layout the TMA would have written; then
//         D += A A^T with A = that tile.  The accumulator goes out once, with its
//         largest diagonal entry.
//   Quad: unit (head h, row tile rt of M16); a stage is the tile of 128 M16 rows
//         (64 neurons, gate and up rows interleaved by 16) and the hi / lo tiles
//         of C~_h; D += A Chi^T + A Clo^T, then every row's m . D[row] in fp32.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(smem_dst)),
               "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Two fp32 values (a packed pair) rounded to fp16 and packed, low half first.
__device__ __forceinline__ uint32_t h2_bits(uint64_t v) {
  const float2 f = unpk(v);
  const __half2 h = __floats2half2_rn(f.x, f.y);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int MODE>
__global__ void __launch_bounds__(kMomentThreads) moment_kernel(const __grid_constant__ CUtensorMap mapA,
                                                                const __grid_constant__ CUtensorMap mapB,
                                                                const MomentParams p) {
  pdl_enter();
  constexpr bool kGram = MODE == kMomentGram;
  constexpr int S = kGram ? kGramStages : kQuadStages;        // TMA stages
  constexpr uint32_t kSB = kGram ? kGramStageBytes : 3 * kMomentTileBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  // stages first (1024-byte aligned); Gram: then 64 floats of 1/r per stage
  uint8_t* st0 = base;
  float* irs0 = reinterpret_cast<float*>(base + (size_t)S * kSB);
  constexpr int NB = kGram ? 1 : 2;   // accumulator buffers (quad: one unit's MMAs beside the last one's epilogue)
  // Gram: full = the TMA copies landed, cvt = the converter warps rewrote the stage, empty =
  // the MMAs read it.  Quad: full, empty.
  __shared__ uint64_t full[S], empty[S], cvt[kGram ? S : 1], tfull[NB], tempty[NB], drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_s;
  __shared__ uint32_t dmax_s;   // Gram: the largest diagonal entry of the unit's block (fp32 bits, >= 0)
  volatile int* abort_flag = &abort_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Gram: one unit per CTA; quad: a persistent grid walks units blockIdx.x, + gridDim.x, ...
  const int ustep = kGram ? p.n_units : (int)gridDim.x;
  const int h = (int)blockIdx.x % p.H, c = (int)blockIdx.x / p.H;
  int kb0 = 0, nkb = p.nkb;
  if (kGram) {
    kb0 = c * p.kpc;
    nkb = p.nkb - kb0 < p.kpc ? p.nkb - kb0 : p.kpc;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      if (kGram) mbar_init(&cvt[s], 4);   // one arrival per converter warp
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);   // one arrival per epilogue warp
    }
    mbar_init(&drain, 1);
    abort_s = 0;
    dmax_s = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&mapA);
    if (!kGram) prefetch_tmap(&mapB);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, 128 * NB);
    tmem_relinquish();
  }
  // Gram: boxes of 32 features per stage; the MMA reads all four, so the ones past
  // ceil(d_head / 32) are zeroed once (the TMA never writes them)
  const int gboxes = kGram ? (p.dh + 31) / 32 : 0;
  if (kGram && warp >= 2 && gboxes < 4) {
    const int per = (4 - gboxes) * kGramBox / 16;   // uint4 per stage
    for (int i = threadIdx.x - 64; i < S * per; i += 128) {
      const int s = i / per, e = i % per;
      reinterpret_cast<uint4*>(st0 + (size_t)s * kSB + (size_t)gboxes * kGramBox)[e] = make_uint4(0, 0, 0, 0);
    }
    fence_async_smem();   // visible to the tensor-core reads
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      int issued = 0;   // stage uses so far (the ring runs on across units)
      for (int u = (int)blockIdx.x; ok && u < p.n_units; u += ustep) {
        const int uh = u % p.H, uc = u / p.H;
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = issued % S;
          const uint32_t ph = (uint32_t)((issued / S) & 1);
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.status)) { ok = false; break; }
          uint8_t* st = st0 + (size_t)s * kSB;
          if constexpr (kGram) {
            // a's columns uh*dh .. + 32*gboxes (past dh: the next head's, or zeros past H*dh)
            mbar_arrive_expect_tx(&full[s], (uint32_t)(gboxes * kGramBox) + 256u);
            for (int bx = 0; bx < gboxes; ++bx)
              tma_load_2d(st + bx * kGramBox, &mapA, &full[s], uh * p.dh + 32 * bx, (kb0 + kb) * 64);
            bulk_load(irs0 + s * 64, p.inv_r + (size_t)(kb0 + kb) * 64, 256u, &full[s]);
          } else {
            mbar_arrive_expect_tx(&full[s], kSB);
            if (p.stream)
              tma_load_2d(st, &mapA, &full[s], uh * p.dh + kb * 64, uc * kMomentRows);
            else
              tma_load_3d(st, &mapA, &full[s], kb * 64, uc * kMomentRows, uh);
            tma_load_2d(st + kMomentTileBytes, &mapB, &full[s], kb * 64, uh * kMomentRows);
            tma_load_2d(st + 2 * kMomentTileBytes, &mapB, &full[s], kb * 64, (p.H + uh) * kMomentRows);
          }
          ++issued;
        }
      }
      if (!ok) {
        // let every copy already issued land before shared memory is released
        const int n = issued < S ? issued : S;
        for (int i = 1; i <= n; ++i) {
          const int q = issued - i;
          volatile int dummy = 0;
          mbar_wait(&full[q % S], (uint32_t)((q / S) & 1), &dummy, p.status, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // Gram: A = B = the stage, MN-major (features along M and N, tokens along K)
      constexpr uint32_t idesc = kGram ? idesc_f16_mn(128, 128, 0) : idesc_f16(128, 128, 0);
      constexpr uint64_t kT = (uint64_t)(kMomentTileBytes >> 4);
      bool ok = true;
      int g = 0;   // stage uses so far (quad)
      for (int u = (int)blockIdx.x, li = 0; ok && u < p.n_units; u += ustep, ++li) {
        const int b = li % NB;
        if constexpr (!kGram) {
          // the buffer's previous unit must have been read out by the epilogue
          if (!mbar_wait(&tempty[b], (uint32_t)(((li / NB) & 1) ^ 1), abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
        }
        const uint32_t d = tmem + (uint32_t)(b * 128);
        for (int kb = 0; kb < nkb; ++kb) {
          if constexpr (kGram) {
            const int s = kb % S;
            if (!mbar_wait(&cvt[s], (uint32_t)((kb / S) & 1), abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint64_t da = smem_desc_mn_sw64(smem_u32(st0 + (size_t)s * kSB), kGramBox);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)   // 16 tokens = 16 rows of 64 B per K slice
              mma_f16_ss(d, da + 64 * ks, da + 64 * ks, idesc, (kb | ks) != 0 ? 1u : 0u);
            mma_commit(&empty[s]);
          } else {
            const int s = g % S;
            if (!mbar_wait(&full[s], (uint32_t)((g / S) & 1), abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint64_t da = smem_desc_k_sw128(smem_u32(st0 + (size_t)s * kSB));
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              mma_f16_ss(d, da + 2 * ks, da + kT + 2 * ks, idesc, (kb | ks) != 0 ? 1u : 0u);
              mma_f16_ss(d, da + 2 * ks, da + 2 * kT + 2 * ks, idesc, 1u);
            }
            mma_commit(&empty[s]);
            ++g;
          }
        }
        if (ok) mma_commit(&tfull[b]);
      }
      if (!ok) {
        mma_commit(&drain);
        volatile int dummy = 0;
        mbar_wait(&drain, 0, &dummy, p.status, 100000000ull);
      }
    }
  } else {
    const int q = warp & 3;              // TMEM lane quarter this warp may read
    const int row = q * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    int w_ok = 1;
    if constexpr (kGram) {
      // ---- converter: each stage rewritten in place, bf16 a -> fp16 a/r.  A 16-byte chunk
      // holds 8 features of one token; the 64-byte swizzle only permutes chunks within a
      // token's 64-byte row, so chunk X of a box belongs to token (X % 256) / 4.
      // An fp16 overflow needs no check here: it becomes inf in the operand, so the
      // head's diagonal is not finite and the reduction latches the range error.
      const int ct = threadIdx.x - 64;   // 0..127
      const int nch = gboxes * (kGramBox / 16);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % S;
        int ok = 1;
        if (lane == 0) ok = mbar_wait(&full[s], (uint32_t)((kb / S) & 1), abort_flag, p.status) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) { w_ok = 0; break; }
        uint4* st = reinterpret_cast<uint4*>(st0 + (size_t)s * kSB);
        const float* irs = irs0 + s * 64;
#pragma unroll 2
        for (int x = ct; x < nch; x += 128) {
          const uint4 w = st[x];
          const float ir = irs[(x & 255) >> 2];
          const uint64_t ir2 = pk(ir, ir);
          uint4 o;
          o.x = h2_bits(mul2(pk_u(w.x << 16, w.x & 0xffff0000u), ir2));
          o.y = h2_bits(mul2(pk_u(w.y << 16, w.y & 0xffff0000u), ir2));
          o.z = h2_bits(mul2(pk_u(w.z << 16, w.z & 0xffff0000u), ir2));
          o.w = h2_bits(mul2(pk_u(w.w << 16, w.w & 0xffff0000u), ir2));
          st[x] = o;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&cvt[s]);
      }
      if (w_ok && lane == 0) w_ok = mbar_wait(&tfull[0], 0, abort_flag, p.status) ? 1 : 0;
      w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
      if (w_ok) {
        tc_fence_after();
        // D[i][j] (i = this lane's feature row) goes to [j][i]: a warp's 32 lanes
        // write 128 contiguous bytes per column.
        float* dst = p.gram + (size_t)(c * p.H + h) * kMomentRows * kMomentRows + row;
        float dg = 0.f;   // D[row][row]; rows past dh are zero
        for (int j0 = 0; j0 < p.dh; j0 += 16) {
          uint32_t v[16];
          tmem_ld16(tl + (uint32_t)j0, v);
          tmem_ld_wait();
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            dst[(size_t)(j0 + jj) * kMomentRows] = __uint_as_float(v[jj]);
            if (j0 + jj == row) dg = __uint_as_float(v[jj]);
          }
        }
        // sums of squares: >= 0, so the fp32 bit patterns order like the values
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dg = fmaxf(dg, __shfl_xor_sync(0xffffffffu, dg, o));
        if (lane == 0) atomicMax(&dmax_s, __float_as_uint(dg));
      }
      // every epilogue warp arrives here, whether or not its waits succeeded
      named_barrier_sync(1, 128);
      if (w_ok && warp == 2 && lane == 0) p.cmax[(size_t)c * p.H + h] = __uint_as_float(dmax_s);
    } else {
      // ---- quad: the units of this CTA, accumulator buffers alternating
      for (int u = (int)blockIdx.x, li = 0; u < p.n_units; u += ustep, ++li) {
        const int b = li % NB;
        int ok = 1;
        if (lane == 0) ok = mbar_wait(&tfull[b], (uint32_t)((li / NB) & 1), abort_flag, p.status) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        const int uh = u % p.H, rt = u / p.H;
        const __half* mrow = p.stream
                                 ? p.M16 + (size_t)(rt * kMomentRows + row) * p.HD + (size_t)uh * p.dh
                                 : p.M16 + ((size_t)uh * 2 * p.I_pad + (size_t)rt * kMomentRows + row) * p.dh;
        const uint32_t tb = tl + (uint32_t)(b * 128);
        float acc = 0.f;
        for (int n0 = 0; n0 < p.dh; n0 += 16) {
          uint32_t v[16];
          tmem_ld16(tb + (uint32_t)n0, v);
          const uint4 m0 = __ldg(reinterpret_cast<const uint4*>(mrow + n0));
          const uint4 m1 = n0 + 8 < p.dh ? __ldg(reinterpret_cast<const uint4*>(mrow + n0 + 8)) : make_uint4(0, 0, 0, 0);
          tmem_ld_wait();
          const __half* e0 = reinterpret_cast<const __half*>(&m0);
          const __half* e1 = reinterpret_cast<const __half*>(&m1);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc = fmaf(__uint_as_float(v[i]), __half2float(e0[i]), acc);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc = fmaf(__uint_as_float(v[8 + i]), __half2float(e1[i]), acc);
        }
        // the buffer is read out: hand it back to the MMA warp
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[b]);
        acc *= p.scale[uh];
        // rows 32q + l (gate) and 32q + 16 + l (up) are neuron 64 rt + 16 q + l
        const float pair = acc + __shfl_xor_sync(0xffffffffu, acc, 16);
        if (lane < 16) p.out[(size_t)uh * p.I_pad + (size_t)rt * 64 + q * 16 + lane] = pair;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128 * NB);
  }
}

size_t moment_smem_bytes(int mode) {
  return 1024 + (mode == kMomentGram ? (size_t)kGramStages * (kGramStageBytes + 256)
                                     : (size_t)kQuadStages * 3 * kMomentTileBytes);
}

cudaError_t launch_moment(const CUtensorMap* maps, const MomentParams& p, cudaStream_t s) {
  if (p.n_units <= 0 || p.nkb <= 0) return cudaErrorInvalidValue;
  const size_t smem = moment_smem_bytes(p.mode);
  cudaError_t e;
  if (p.mode == kMomentGram) {
    auto* fn = moment_kernel<kMomentGram>;
    if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
      return e;
    // two CTAs per SM need the largest shared-memory carve-out
    if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  (int)cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
      return e;
    if (cudaError_t e_ = launch_pdl(fn, p.n_units, kMomentThreads, smem, s, maps[0], maps[1], p); e_ != cudaSuccess)
      return e_;
  } else if (p.mode == kMomentQuad) {
    if (p.nkb > kQuadStages) return cudaErrorInvalidValue;
    auto* fn = moment_kernel<kMomentQuad>;
    if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
      return e;
    const int grid = p.ctas > 0 && p.ctas < p.n_units ? p.ctas : p.n_units;
    if (cudaError_t e_ = launch_pdl(fn, grid, kMomentThreads, smem, s, maps[0], maps[1], p); e_ != cudaSuccess)
      return e_;
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_inv_r(const uint16_t* x, float* inv_r, int T, int n_pad, int D, float eps, int sm_count,
                        cudaStream_t s) {
  int blocks = (n_pad + 15) / 16;   // 8 warps, two tokens each
  if (blocks > 8 * sm_count) blocks = 8 * sm_count;
  if (cudaError_t e_ = launch_pdl(inv_r_kernel, blocks, 256, 0, s, x, inv_r, T, n_pad, D, eps); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

cudaError_t launch_gram_reduce(const float* gram, const float* cmax, __half* CC, float* scale, int n_chunks, int H,
                               int dh, uint32_t* status, const uint16_t* a, const float* inv_r, int T, DevScales* sc,
                               cudaStream_t s) {
  if (cudaError_t e_ = launch_pdl(gram_reduce_kernel, dim3(H, 128 / kReduceRows), 256, 0, s, gram, cmax, CC, scale,
                                  n_chunks, H, dh, status, a, inv_r, T, sc); e_ != cudaSuccess)
    return e_;
  if (cudaError_t e = cudaGetLastError(); e != cudaSuccess) return e;
  if (cudaError_t e_ = launch_pdl(moment_fallback_kernel, H, 1024, 0, s, a, inv_r, T, H, dh, CC, scale, sc, status); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

cudaError_t launch_moment_finalize(const float* out, int T, int H, int G, int I, int I_pad, float* S_out,
                                   float* S_head_out, const DevScales* sc, int D, cudaStream_t s) {
  if (cudaError_t e_ = launch_pdl(moment_finalize_kernel, dim3((I + 255) / 256, G), 256, 0, s, out, T, H, G, I, I_pad,
                                  S_out, S_head_out, sc, D); e_ != cudaSuccess)
    return e_;
  return cudaGetLastError();
}

}  // namespace aff
