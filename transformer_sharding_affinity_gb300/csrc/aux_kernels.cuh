// aux_kernels.cuh -- host-side launchers of the auxiliary kernels.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "scales.cuh"

namespace aff {

// n16 = gamma x / r 2^e_n, a16 = a / r (max recorded in sc->amax), inv_r = 1 / r.
cudaError_t launch_prep_tokens(const uint16_t* x, const uint16_t* a, const uint16_t* gamma, __half* n16, __half* a16,
                               float* inv_r, int T, int D, int HD, float eps, uint32_t* status, int sm_count,
                               DevScales* sc, cudaStream_t s);
// a16 staged again as a / r 2^e_a when sc->amax calls for it (else returns at once).
cudaError_t launch_restage_a(const uint16_t* a, const float* inv_r, __half* a16, int T, int HD, const DevScales* sc,
                             uint32_t* status, int sm_count, cudaStream_t s);
// W16 (as launch_prep_gate_up) and gamma*Wo^T hi / lo ([HD][2][D]) in one launch, both
// unscaled, recording the maxima of DevScales.
cudaError_t launch_weight_stage(const uint16_t* Wg, const uint16_t* Wu, __half* W16, int I, int I_pad, int D,
                                const uint16_t* Wo, const uint16_t* gamma, __half* GWo16, int HD, DevScales* sc,
                                int sm_count, cudaStream_t s);
// W16 ([I_pad / 16][2][16][D], gate and up rows of 16 neurons), unscaled; records sc->wmax.
cudaError_t launch_prep_gate_up(const uint16_t* Wg, const uint16_t* Wu, __half* W16, int I, int I_pad, int D,
                                DevScales* sc, cudaStream_t s);
// W16, GWo16 (when given) and Wo16 (when given) staged again at their power-of-two scales
// when the recorded maxima call for it; otherwise returns at once.
cudaError_t launch_weight_restage(const uint16_t* Wg, const uint16_t* Wu, __half* W16, int I, int I_pad, int D,
                                  const uint16_t* Wo, const uint16_t* gamma, __half* GWo16, __half* Wo16, int HD,
                                  DevScales* sc, uint32_t* status, int sm_count, cudaStream_t s);
cudaError_t launch_wd_colnorm(const uint16_t* Wd, float* wdn, int D, int I, int I_pad, cudaStream_t s);
cudaError_t launch_wd_colnorm_f32(const float* Wd, float* wdn, int D, int I, cudaStream_t s);
cudaError_t launch_reduce_partials(const float* partial, double* out, int n_chunks, int halves, int H, int I_pad,
                                   cudaStream_t s);
// The partial sums carry the head operands' 2^2(e_m + e_a) (scales.cuh), removed here.
cudaError_t launch_reduce_finalize(const float* partial, const float* wdn, int fo, int n_chunks, int groups, int T,
                                   int H, int G, int I, int I_pad, float* S_out, float* S_head_out,
                                   const DevScales* sc, int D, cudaStream_t s);
cudaError_t launch_finalize_up(const double* sh, const float* wdn, int fo, int T, int H, int G, int I, int I_pad,
                               float* S_out, float* S_head_out, cudaStream_t s);
cudaError_t launch_wait_selftest(uint32_t* status, unsigned long long limit_ns, cudaStream_t s);
cudaError_t launch_to_fp16(const uint16_t* in, __half* out, size_t n, uint32_t* status, cudaStream_t s);
cudaError_t launch_loo_rho(const float* cn, const float* inv_r, float* rho, int T, int T_pad, int H, int D,
                           int groups, const DevScales* sc, cudaStream_t s);
cudaError_t launch_prep_wd(const uint16_t* Wd, __half* Wd16, __half* WdT16, int D, int I, int I_pad, uint32_t* status,
                           cudaStream_t s);
cudaError_t launch_prep_qkv(const uint16_t* Wq, const uint16_t* Wk, const uint16_t* Wv, const uint16_t* gamma_next,
                            __half* out, int G, int hpg, int dh, int D, uint32_t* status, cudaStream_t s);
cudaError_t launch_down_token_weights(const __half* alpha16, const float* ssx, float* cpart, int T, int T_pad, int D,
                                      int I_pad, int chunk, float eps, int groups, cudaStream_t s);
cudaError_t launch_finalize_down(const float* cpart, const float* bnorm, int n_chunks, int bhalves, int T, int I,
                                 int I_pad, int G, float* S_out, cudaStream_t s);

struct F32UpArgs {
  const float *a, *x, *Wo, *gamma, *Wg, *Wu;
  float *n32, *a32, *M32, *partial;
  float2* ab;
  int T, D, H, dh, I, n_chunks, chunk, fo;
  float eps;
};
cudaError_t launch_f32_up(const F32UpArgs& A, cudaStream_t s);

struct F32DownArgs {
  const float *x, *gamma, *Wg, *Wu, *Wd, *gamma_next, *Wq, *Wk, *Wv;
  float *n32, *alpha32, *ssx, *cpart, *bnorm;
  int T, D, H, G, dh, I, n_chunks, chunk;
  float eps;
};
cudaError_t launch_f32_down(const F32DownArgs& A, cudaStream_t s);

}  // namespace aff
