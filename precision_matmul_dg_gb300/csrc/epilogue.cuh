// Fused epilogue of the GEMM: t = alpha*acc + beta*C + bias, then GELU.
//
// Order and form follow the "DeepGEMM" articles' epilogue generator
// (kwkr.cn/news/562171, section 2.2 third layer: alpha * gemm_out + beta * ...,
// bias + GELU fused with no intermediate written back; discosf.com/news/5532976,
// section 6.1, op_type "gelu"): the bias is added after alpha/beta and before
// the activation, and GELU is the exact erf form.  Arithmetic is FP32; the
// result is rounded once to FP16 (round to nearest even).
#pragma once

#include <cuda_fp16.h>

namespace dg {

__device__ __forceinline__ float gelu_erf(float t) {
  return 0.5f * t * (1.0f + erff(t * 0.70710678118654752f));
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
