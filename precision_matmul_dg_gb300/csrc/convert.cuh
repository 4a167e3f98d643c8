// Exact widening of narrow operands to FP16, shared by the kernels that read
// int8 values or packed E2M1 codes.  Every int8 value (|v| <= 128) and every
// E2M1 value ({0, .5, 1, 1.5, 2, 3, 4, 6} and their negatives) is exactly
// representable in FP16, so these conversions change no value.  Codes are
// packed two a byte, k = 2p in the low nibble of byte p (discosf.com/news/
// 5532976, section 4.3 packing), the order cvt.rn.f16x2.e2m1x2 reads them in.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace dg {

// Two int8 values (the low two bytes of `two_bytes`) as an FP16 pair: byte
// b becomes the FP16 bits 0x6400 | (b ^ 0x80) = 1024 + (v + 128), and 1152
// is subtracted, exactly.
__device__ __forceinline__ uint32_t i8x2_to_f16x2(uint32_t two_bytes) {
  const uint32_t x = (two_bytes ^ 0x8080u);
  uint32_t a = __byte_perm(x, 0x64646464u, 0x4140);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  __half2 h = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Eight E2M1 codes (the four bytes of `w`) as four FP16 pairs, byte i into
// pair i with its low nibble in the low half: the word is split into its
// bytes once and each byte goes through the hardware pair conversion.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t* f) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(f[0]), "=r"(f[1]), "=r"(f[2]), "=r"(f[3])
      : "r"(w));
}

__device__ __forceinline__ uint4 e2m1x8_to_f16x8(uint32_t w) {
  uint32_t f[4];
  e2m1x8_to_f16x2x4(w, f);
  return make_uint4(f[0], f[1], f[2], f[3]);
}

}  // namespace dg
