// Fused epilogue of the GEMM: t = alpha*acc + beta*C + bias, then GELU.
//
// Order and form follow the "DeepGEMM" articles' epilogue generator
// (kwkr.cn/news/562171, section 2.2 third layer: alpha * gemm_out + beta * ...,
// bias + GELU fused with no intermediate written back; discosf.com/news/5532976,
// section 6.1, op_type "gelu"): the bias is added after alpha/beta and before
// the activation, and GELU is the erf form (evaluated to 1e-7 relative, see
// gelu_erf).  Arithmetic is FP32; the result is rounded once to FP16 (round to
// nearest even).
#pragma once

#include <cuda_fp16.h>

namespace dg {

// GELU(t) = t * Phi(t), Phi the standard normal CDF, written as
// Phi(t) = 1 - q for t >= 0 and q for t < 0, with q = erfc(|t| / sqrt 2) / 2.
// erfc(z), z >= 0, is the rational-exponential approximation of Abramowitz &
// Stegun, Handbook of Mathematical Functions, eq. 7.1.26 (after Hastings):
//   erfc(z) = (a1 s + a2 s^2 + a3 s^3 + a4 s^4 + a5 s^5) exp(-z^2) + e(z),
//   s = 1 / (1 + p z),  |e(z)| <= 1.5e-7,
// so |GELU error| <= 1e-7 |t| plus FP32 rounding: far inside the 2^-10
// relative budget, at one reciprocal, one exponential and five FMAs.
__device__ __forceinline__ float gelu_erf(float t) {
  constexpr float p = 0.3275911f, a1 = 0.254829592f, a2 = -0.284496736f, a3 = 1.421413741f,
                  a4 = -1.453152027f, a5 = 1.061405429f;
  const float z = fabsf(t) * 0.70710678118654752f;
  const float s = __fdividef(1.0f, fmaf(p, z, 1.0f));
  const float poly = fmaf(fmaf(fmaf(fmaf(a5, s, a4), s, a3), s, a2), s, a1) * s;
  const float q = 0.5f * poly * __expf(-z * z);
  return t * (t >= 0.0f ? 1.0f - q : q);
}

struct Epi {
  float alpha, beta;
  int flags;  // kEpiBias | kEpiGelu
};

// t for one element; c and b are the C and bias values (0 when unused).
__device__ __forceinline__ float epi_apply(float acc, float c, float b, const Epi& e) {
  float t = e.alpha * acc;
  t = fmaf(e.beta, c, t);
  t += b;
  if (e.flags & 2) t = gelu_erf(t);
  return t;
}

}  // namespace dg
