// Widening pre-pass: int8 or packed E2M1 operand -> FP16, exactly.
//
// For compute-bound shapes the INT8 and W4A16 GEMMs widen their narrow
// operands once into an FP16 copy (a library-owned workspace) and run the
// FP16 tensor-core kernel, instead of widening every tile in shared memory
// for every output tile that reads it (which makes those kernels shared-
// memory-bandwidth bound).  Memory-bound shapes keep the in-kernel widening.
//
// Every int8 value and every E2M1 code is exactly representable in FP16
// (|int8| <= 128; E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}), so the copy
// changes no value.  Codes are read two per byte, k = 2p in the low nibble of
// byte p (discosf.com/news/5532976, section 4.3 packing; the nibble order is
// the same one cvt.rn.f16x2.e2m1x2 uses).
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace dg {
namespace {

__device__ __forceinline__ uint32_t i8x2_to_f16x2(uint32_t two_bytes) {
  // byte b -> fp16 bits 0x6400 | (b ^ 0x80) = 1024 + (v + 128); minus 1152
  const uint32_t x = (two_bytes ^ 0x8080u);
  uint32_t a = __byte_perm(x, 0x64646464u, 0x4140);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  __half2 h = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t o;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
      : "=r"(o)
      : "r"(byte));
  return o;
}

// int8 [rows x ld_src] -> fp16 [rows x ld_dst]; 16 source bytes per thread step.
// Reads whole 16-byte groups up to the row pitch (a multiple of 16 bytes);
// columns >= K of the copy are never read by the GEMM.
__global__ void widen_i8_kernel(const int8_t* __restrict__ src, int64_t rows, int64_t groups,
                                int64_t ld_src, __half* __restrict__ dst, int64_t ld_dst) {
  const int64_t total = rows * groups;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / groups, g = i - r * groups;
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(src + r * ld_src + g * 16));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    uint4 o[2];
    uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      ow[2 * q] = i8x2_to_f16x2(ws[q] & 0xFFFFu);
      ow[2 * q + 1] = i8x2_to_f16x2(ws[q] >> 16);
    }
    uint4* d = reinterpret_cast<uint4*>(dst + r * ld_dst + g * 16);
    d[0] = o[0];
    d[1] = o[1];
  }
}

// packed E2M1 [rows x ld_src bytes] -> fp16 [rows x ld_dst]; 16 bytes = 32
// codes per thread step.
__global__ void widen_e2m1_kernel(const uint8_t* __restrict__ src, int64_t rows, int64_t groups,
                                  int64_t ld_src_bytes, __half* __restrict__ dst, int64_t ld_dst) {
  const int64_t total = rows * groups;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / groups, g = i - r * groups;
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(src + r * ld_src_bytes + g * 16));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    uint4* d = reinterpret_cast<uint4*>(dst + r * ld_dst + g * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 o;
      o.x = e2m1x2_to_f16x2(ws[q] & 0xFFu);
      o.y = e2m1x2_to_f16x2((ws[q] >> 8) & 0xFFu);
      o.z = e2m1x2_to_f16x2((ws[q] >> 16) & 0xFFu);
      o.w = e2m1x2_to_f16x2(ws[q] >> 24);
      d[q] = o;
    }
  }
}

int grid_for(int64_t items, int sm_count) {
  int64_t blocks = (items + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count) * 16;
  if (blocks > cap) blocks = cap;
  return static_cast<int>(blocks < 1 ? 1 : blocks);
}

}  // namespace

int64_t widened_ld(int64_t K) { return (K + 31) / 32 * 32; }

cudaError_t launch_widen(dg_dtype dtype, const void* src, int64_t rows, int64_t K, int64_t ld_src,
                         __half* dst, cudaStream_t stream, int sm_count) {
  const int64_t ld_dst = widened_ld(K);
  if (dtype == DG_I8) {
    const int64_t groups = (K + 15) / 16;  // 16 int8 per group; ld_src is a multiple of 16
    widen_i8_kernel<<<grid_for(rows * groups, sm_count), 256, 0, stream>>>(
        static_cast<const int8_t*>(src), rows, groups, ld_src, dst, ld_dst);
  } else if (dtype == DG_E2M1) {
    const int64_t groups = ((K + 1) / 2 + 15) / 16;  // 32 codes per group; pitch ld_src/2 bytes
    widen_e2m1_kernel<<<grid_for(rows * groups, sm_count), 256, 0, stream>>>(
        static_cast<const uint8_t*>(src), rows, groups, ld_src / 2, dst, ld_dst);
  } else {
    return cudaErrorInvalidValue;
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dg
