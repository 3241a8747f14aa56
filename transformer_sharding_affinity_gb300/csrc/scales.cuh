// scales.cuh -- power-of-two rescaling of the fp16 tensor-core operands.
//
// The bf16 path stages its tensor-core operands in fp16, whose range
// (|v| < 65504, normal above 2^-14) is far narrower than bf16's.  To accept
// every finite bf16 input, each staged tensor is multiplied by a power of two
// 2^e chosen from a device-side maximum, and the fp32 results are multiplied
// by the inverse power afterwards.  Scaling by a power of two commutes with
// rounding (away from the subnormal range), so a result is the same as with
// no scaling whenever no operand would have overflowed or been subnormal.
//
//   weights  W16 = [Wg; Wu] 2^e_w, GWo16 = gamma Wo^T 2^e_g, Wo16 = Wo 2^e_o:
//            staged unscaled while their largest magnitudes are recorded,
//            then staged again (weight_restage_kernel) only when a maximum
//            lies outside [2^-6, 2^15), so ordinary weights pay for one small
//            launch;
//   fold     M16 = M 2^e_m, e_m from the bound
//            |M[k][j]| <= D max|W| max|gamma_d Wo[d][j]|;
//   n16      gamma x / r * 2^e_n, from the bound |x_d| / r <= sqrt(D);
//   a16      a / r * 2^e_a, from the largest staged |a / r|: 0 unless that
//            maximum lies outside [2^-6, 2^15), in which case a16 is staged
//            again.
// The maxima live in DevScales inside the workspace; every consumer derives
// the exponents from them with the same functions, so all kernels agree.
#pragma once

#include <cstdint>

namespace aff {

struct DevScales {
  uint32_t wmax;    // max over Wg and Wu of |value| (fp32 bits; atomicMax over non-negative floats)
  uint32_t womax;   // max |Wo|
  uint32_t gwmax;   // max |gamma_d Wo[d][j]|
  uint32_t gmax;    // max |gamma| recorded by the token side (the scale of n16)
  uint32_t amax;    // max |a_t / r_t| as first staged (FO, LOO, ADD direct)
  uint32_t amax2;   // second-moment ADD fallback: max |a_t / r_t| over every token
  uint32_t redo;    // second-moment ADD: 1 when the Gram matrices are recomputed with a scale
  uint32_t units;   // head passes (FO, LOO, direct ADD): units claimed so far by the tile kernel's CTAs
};

constexpr int kScaleTarget = 13;   // a normalised maximum lands in [2^13, 2^14)
constexpr int kScaleClamp = 60;    // |exponent| limit, so that combined factors stay finite in fp32

// Exponent e with m * 2^e in [2^13, 2^14) for a finite m > 0, else 0; clamped.
__host__ __device__ inline int scale_exp_norm(float m) {
  if (!(m > 0.f) || !(m <= 3.4e38f)) return 0;
  int e2 = 0;
  // floor(log2(m)) without libm: the fp32 exponent field (m is normal here or a subnormal
  // handled below)
  uint32_t bits;
  __builtin_memcpy(&bits, &m, 4);
  const int ex = (int)((bits >> 23) & 0xFF);
  if (ex == 0) {
    e2 = -127;   // subnormal: below 2^-126
  } else {
    e2 = ex - 127;
  }
  int e = kScaleTarget - e2;
  if (e > kScaleClamp) e = kScaleClamp;
  if (e < -kScaleClamp) e = -kScaleClamp;
  return e;
}

// Activations: 0 while m is in [2^-6, 2^15), else normalised.
__host__ __device__ inline int scale_exp_act(float m) {
  if (m >= 0.015625f && m < 32768.f) return 0;
  return scale_exp_norm(m);
}

// 2^e as fp32 for |e| <= 126, built from the exponent field (exact).
__host__ __device__ inline float pow2f(int e) {
  const uint32_t bits = (uint32_t)(e + 127) << 23;
  float f;
  __builtin_memcpy(&f, &bits, 4);
  return f;
}

__host__ __device__ inline float bits_f(uint32_t b) {
  float f;
  __builtin_memcpy(&f, &b, 4);
  return f;
}

__host__ __device__ inline int clamp_exp(int e) {
  return e > kScaleClamp ? kScaleClamp : (e < -kScaleClamp ? -kScaleClamp : e);
}

// The exponents every consumer uses, from the recorded maxima.  Sums of two
// clamped exponents stay within fp32's exponent range.
struct ScaleExps {
  int e_w, e_g, e_m, e_o, e_n, e_a;
};

__host__ __device__ inline ScaleExps scale_exps(const DevScales& s, int D) {
  ScaleExps x;
  // ceil(log2(D)): D <= 2^lgD
  int lgD = 0;
  while ((int64_t)1 << lgD < (int64_t)D) ++lgD;
  x.e_w = scale_exp_act(bits_f(s.wmax));
  x.e_g = scale_exp_act(bits_f(s.gwmax));
  x.e_o = scale_exp_act(bits_f(s.womax));
  // |M[k][j]| <= D max|W| max|gamma Wo|: the bound's product could leave fp32's range, so
  // its factors' normalising exponents are combined instead (each factor times its 2^e
  // lies in [2^13, 2^14))
  x.e_m = clamp_exp(scale_exp_norm(bits_f(s.wmax)) + scale_exp_norm(bits_f(s.gwmax)) - 14 - lgD);
  // |gamma_d x_d / r| <= max|gamma| sqrt(D) (x_d^2 <= D mean(x^2) <= D r^2); sqrt(D) <= 2^lg
  int lg = 0;
  while ((int64_t)1 << (2 * lg) < (int64_t)D) ++lg;
  x.e_n = clamp_exp(scale_exp_norm(bits_f(s.gmax)) - lg);
  x.e_a = scale_exp_act(bits_f(s.amax));
  return x;
}

}  // namespace aff
