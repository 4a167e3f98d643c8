// Fused epilogue of the GEMM: t = alpha*acc + beta*C + bias, then GELU; or
// t = alpha*acc + beta*C, then a program of ops.
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

#include "internal.h"

namespace dg {

// GELU(t) = t * Phi(t), Phi the standard normal CDF, written as
// Phi(t) = 1 - q for t >= 0 and q for t < 0, with q = erfc(|t| / sqrt 2) / 2.
// erfc(z), z >= 0, is the rational-exponential approximation of Abramowitz &
// Stegun, Handbook of Mathematical Functions, eq. 7.1.26 (after Hastings):
//   erfc(z) = (a1 s + a2 s^2 + a3 s^3 + a4 s^4 + a5 s^5) exp(-z^2) + e(z),
//   s = 1 / (1 + p z),  |e(z)| <= 1.5e-7,
// so |GELU error| <= 1e-7 |t| plus FP32 rounding: far inside the 2^-10
// relative budget, at one reciprocal, one exponential and five FMAs.
// z = |t| / sqrt 2 and the 1/2 of q are folded into the constants, and
// exp(-z^2) = 2^(-t^2 log2(e) / 2) goes straight to the hardware base-2
// exponential, so a value costs about 14 instructions.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float gelu_erf(float t) {
  constexpr float p = 0.3275911f, a1 = 0.254829592f, a2 = -0.284496736f, a3 = 1.421413741f,
                  a4 = -1.453152027f, a5 = 1.061405429f;
  constexpr float kP = p * 0.70710678118654752f;  // p / sqrt 2
  constexpr float kE = -0.72134752044448170f;      // -log2(e) / 2
  const float s = __fdividef(1.0f, fmaf(kP, fabsf(t), 1.0f));
  const float half_poly =
      fmaf(fmaf(fmaf(fmaf(0.5f * a5, s, 0.5f * a4), s, 0.5f * a3), s, 0.5f * a2), s, 0.5f * a1) *
      s;
  const float q = half_poly * ex2_approx(t * t * kE);
  const float tq = t * q;
  return t >= 0.0f ? t - tq : tq;
}

// Output quantization (kOpQuantI8, the program's last op): x = a * t rounded
// half to even and saturated to [-128, 127]; NaN gives 0.
__device__ __forceinline__ int8_t quant_i8(float x) {
  if (x != x) return 0;
  return static_cast<int8_t>(__float2int_rn(fminf(fmaxf(x, -128.0f), 127.0f)));
}

// Epilogue ops of a program (dg_epilogue_op in dg.h), applied in order to
// t = alpha * acc + beta * C: the post-processing steps the pages' epilogue
// generator fuses into the GEMM (kwkr.cn/news/562171, section 2.2 third
// layer: bias add, ReLU, quantize-style scaling; GELU as op_type "gelu",
// discosf.com/news/5532976, section 6.1).
// Kept to 16 bytes: every kernel carries it in its parameter struct, and
// those structs stay within 128 bytes (measured on GB300: a by-value
// parameter struct above 128 bytes slowed the streaming GEMV by 10% and the
// tensor-core kernel by 8%).  The ops travel in their own parameter.
struct Epi {
  float alpha, beta;
  int flags;  // kEpiBias | kEpiGelu (bias, then GELU), or kEpiProgram (+ kEpiBias if a bias op)
  int n_ops;  // kEpiProgram: the program's ops [0, n_ops) in order
};

// A program's ops: a kernel parameter of its own (__grid_constant__).
struct EpiProgram {
  EpiOp ops[kMaxEpiOps];
};

// The program's ops on t; b is the column's bias (0 without a bias op).
// ReLU and clamp ignore NaN the way fmaxf / fminf do.
__device__ __forceinline__ float epi_program(float t, float b, const Epi& e,
                                             const EpiProgram& prog) {
#pragma unroll 1
  for (int k = 0; k < e.n_ops; ++k) {
    const EpiOp op = prog.ops[k];
    switch (op.type) {  // kOpScale: t *= a; kOpClamp: t = min(max(t, a), b)
      case kOpBias: t += b; break;
      case kOpRelu: t = t > 0.0f ? t : 0.0f; break;
      case kOpGelu: t = gelu_erf(t); break;
      case kOpScale: t *= op.a; break;
      case kOpClamp: t = fminf(fmaxf(t, op.a), op.b); break;
      default: break;  // kOpQuantI8 is applied by the store (epi_store)
    }
  }
  return t;
}

// t for one element; c and b are the C and bias values (0 when unused).
__device__ __forceinline__ float epi_apply(float acc, float c, float b, const Epi& e,
                                           const EpiProgram& prog) {
  float t = e.alpha * acc;
  t = fmaf(e.beta, c, t);
  if (e.flags & kEpiProgram) return epi_program(t, b, e, prog);
  t += b;
  if (e.flags & kEpiGelu) t = gelu_erf(t);
  return t;
}

// Stores t as element idx of D: FP16 (round to nearest even), or the int8
// code of the program's closing quantization.
__device__ __forceinline__ void epi_store(void* D, int64_t idx, float t, const Epi& e,
                                          const EpiProgram& prog) {
  if (e.flags & kEpiOutI8)
    static_cast<int8_t*>(D)[idx] = quant_i8(prog.ops[e.n_ops - 1].a * t);
  else
    static_cast<__half*>(D)[idx] = __float2half_rn(t);
}

// The kernels' view of a call's scalars and epilogue.
inline Epi make_epi(const GemmArgs& a) { return Epi{a.alpha, a.beta, a.epi, a.n_ops}; }

inline EpiProgram make_program(const GemmArgs& a) {
  EpiProgram p;
  for (int k = 0; k < kMaxEpiOps; ++k) p.ops[k] = k < a.n_ops ? a.ops[k] : EpiOp{0, 0.0f, 0.0f};
  return p;
}

}  // namespace dg
