// moment_kernel.cuh -- the ADD score through each head's second moment of a_h / r.
//
// ADD (paper "Affinity-Aware Sharding for Delayed Tensor Parallelism", §3
// "Affinity scores") is S_hk = E_t[(p_h.w^g_k)^2 + (p_h.w^u_k)^2].  With
// p_h.w = a~_h . m (a~_h = a_h / r, m = the folded row of M_h = W diag(gamma)
// W_o^(h)), every term is a quadratic form of one d_head x d_head matrix:
//   sum_t (a~_t . m)^2 = m^T C_h m,   C_h = sum_t a~_t a~_t^T.
// So instead of contracting every token with every neuron row (T x 2I x d_head
// multiply-adds per head) the pass forms C_h once (T x d_head^2, a tensor-core
// Gram matrix over the tokens) and then evaluates 2I quadratic forms (2I x
// d_head^2, again on the tensor cores).  Same sum, different rounding order.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "scales.cuh"

namespace aff {

enum MomentMode : int {
  kMomentGram = 0,   // C_h partial sums: per (head, token chunk), A = B = a~^T, 128 feature rows x 64 tokens
  kMomentQuad = 1    // per (head, 128 M_h rows): D = M_h C~_h (hi + lo parts), then m . D row by row
};

constexpr int kMomentRows = 128;                          // feature rows of a Gram tile, M_h rows of a quad tile
constexpr int kMomentTileBytes = 128 * 64 * 2;            // one 128-row x 64-element fp16 tile
// Gram stage: 64 tokens of one head's columns of a, as up to four TMA boxes of 32
// features x 64 tokens (64-byte rows, 64-byte swizzle), 4 KB each; the converter
// warps rewrite them in place as fp16 a/r, which the MMA reads as MN-major operands.
constexpr int kGramStages = 6;
constexpr int kGramBox = 64 * 32 * 2;
constexpr int kGramStageBytes = 4 * kGramBox;
constexpr int kQuadStages = 2;                            // d_head <= 128: at most two K blocks
constexpr int kMomentThreads = 192;                       // TMA warp, MMA warp, 4 epilogue warps
// Units of the Gram pass: H x chunks with at most this many CTAs (two per SM on
// 152 SMs, one wave); a function of the shape only, so results do not depend
// on the device.
constexpr int kGramUnits = 304;

struct MomentParams {
  int32_t mode;
  int32_t n_units;
  int32_t H, dh, HD, I_pad;
  int32_t nkb;       // Gram: 64-token K blocks in all, ceil(T / 64); quad: K blocks over d_head
  int32_t kpc;       // Gram: K blocks per token chunk
  int32_t stream;    // quad: M16 is [2 I_pad][H*dh] (else [H][2 I_pad][dh])
  int32_t ctas;      // quad: CTAs of the persistent grid (<= n_units; two fit on an SM)
  uint32_t* status;
  float* gram;       // Gram output: [chunk][H][128 (column j)][128 (row i)] fp32
  float* cmax;       // Gram output: [chunk][H] the block's largest diagonal entry
  const float* inv_r;   // Gram: 1/r per token, [nkb * 64] (0 past T)
  const float* scale;   // quad: per-head scale s_h of the staged C~_h = C_h / s_h
  const __half* M16;    // quad epilogue: the rows it contracted, read again as fp16
  float* out;           // quad output: [H][I_pad], m_g^T C_h m_g + m_u^T C_h m_u (token sums)
};

// Gram chunking of ceil(T / 64) K blocks over H heads.
struct GramSplit {
  int nkb, kpc, n_chunks;
};
inline GramSplit gram_split(int64_t T, int64_t H) {
  GramSplit g;
  g.nkb = (int)((T + 63) / 64);
  int64_t want = H >= kGramUnits ? 1 : kGramUnits / H;
  if (want > g.nkb) want = g.nkb;
  if (want < 1) want = 1;
  g.kpc = (int)((g.nkb + want - 1) / want);
  g.n_chunks = (g.nkb + g.kpc - 1) / g.kpc;
  return g;
}

size_t moment_smem_bytes(int mode);
cudaError_t launch_moment(const CUtensorMap* maps, const MomentParams& p, cudaStream_t s);
// inv_r[t] = 1 / sqrt(mean_d x_t,d^2 + eps) for t < T, 0 for T <= t < n_pad.
cudaError_t launch_inv_r(const uint16_t* x, float* inv_r, int T, int n_pad, int D, float eps, int sm_count,
                         cudaStream_t s);
// C_h = sum over chunks of the Gram partials (in chunk order); s_h = the sum over
// chunks of their largest diagonal entries (>= max_i C_h[i][i]; 1 when not
// positive); CC = [hi; lo] fp16 parts of C_h / s_h: [2][H][128][128], zero
// outside d_head x d_head.  When the unscaled fp16 Gram pass overflowed or lost
// its operands to fp16 subnormals, a second kernel recomputes C_h with a
// power-of-two scale instead (and scale[h] removes it); it returns at once
// otherwise.
cudaError_t launch_gram_reduce(const float* gram, const float* cmax, __half* CC, float* scale, int n_chunks, int H,
                               int dh, uint32_t* status, const uint16_t* a, const float* inv_r, int T, DevScales* sc,
                               cudaStream_t s);
// S_head[h][k] = out[h][k] / T (the folded rows' 2^2e_m removed), S_up[g][k] = sum of
// S_head over g's heads (fp64, head order).
cudaError_t launch_moment_finalize(const float* out, int T, int H, int G, int I, int I_pad, float* S_out,
                                   float* S_head_out, const DevScales* sc, int D, cudaStream_t s);

}  // namespace aff
