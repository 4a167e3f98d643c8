// Block-scaled 4-bit operands (MXFP4): quantization of FP16 rows, and the
// exact widening of MXFP4 operands to BF16 for the tensor-core kernel.
//
// Format (the MX block format; the pages -- discosf.com/news/5532976,
// section 2.2 layer 2 and section 4.3 -- ask for low-bit operands in the
// tensor cores' own formats but fix no block layout): along K, each block of
// 32 values shares one E8M0 scale byte e (X = 2^(e - 127), e = 255 is NaN)
// and each value is an E2M1 code, packed two per byte with k = 2p in the low
// nibble of byte p (the packing of the E2M1 weights).
//
// Quantization (one block of 32 values, one thread):
//   amax   -- the largest magnitude, taken on the FP16 bit patterns (sign
//             cleared; an unsigned maximum orders finite values by magnitude
//             and puts infinities and NaNs above all of them);
//   scale  -- s = floor(log2(amax)) - 2, read off amax's exponent field (or,
//             for an FP16 subnormal, its leading mantissa bit); e = s + 127;
//             an all-zero block takes s = -127; a block with an infinity or
//             a NaN takes e = 255 and codes 0;
//   codes  -- v * 2^-s, exact in FP32, rounded to E2M1 by the conversion
//             instruction (nearest, ties to even, saturating at 6), which
//             keeps the sign of -0 and of negative values that round to 0.
//
// Widening: e2m1(code) has at most two significant bits and e spans 2^-127 ..
// 2^127, so e2m1(code) * X is exact in FP32 and again in BF16 (FP32's
// exponent range; BF16 subnormals reach 2^-133) up to e = 251; above that the
// largest codes overflow to infinities.  The copy is laid out as the FP16
// widening's copies are: rows of widened_ld(K) = 32 * ceil(K / 32) values.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace dg {
namespace {

constexpr int kMxThreads = 256;
constexpr int kMxBlock = 32;  // values per scale

// ---------------------------------------------------------------------------
// Quantization
// ---------------------------------------------------------------------------

// Eight FP32 values -> four bytes of E2M1 codes (value 2i in the low nibble
// of byte i), nearest with ties to even, saturated to the largest finite
// code.  The conversion keeps the sign of negative values that round to zero
// (code 8, -0), as the format's rounding asks (checked on GB300 for -0,
// -1e-30, -0.1 and -0.2499).
__device__ __forceinline__ uint32_t e2m1x8_from_f32(const float (&v)[8]) {
  uint32_t out;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(out)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return out;
}

// 16-byte read-only load.
__device__ __forceinline__ uint4 ld_nc16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Quantizes one block of 32 values held by one thread (`w`: the FP16 values
// as 16 words, zeros past K).  Returns the 16 bytes of codes and sets the
// scale byte.
__device__ __forceinline__ uint4 quantize_block(const uint32_t (&w)[16], uint32_t& scale_byte) {
  uint32_t m = 0;
#pragma unroll
  for (int q = 0; q < 16; ++q) m = __vmaxu2(m, w[q] & 0x7FFF7FFFu);
  const uint32_t amax = max(m & 0xFFFFu, m >> 16);
  if (amax >= 0x7C00u) {
    scale_byte = 255;  // infinity or NaN in the block: codes 0
    return make_uint4(0u, 0u, 0u, 0u);
  }
  int s = -127;  // all-zero block
  if (amax != 0) {
    const int e = static_cast<int>(amax >> 10);
    const int fl = e != 0 ? e - 15 : (31 - __clz(static_cast<int>(amax))) - 24;
    s = fl - 2;
  }
  scale_byte = static_cast<uint32_t>(s + 127);
  // 2^-s as FP32 bits (s in [-26, 13] for a non-zero block; 2^127 for the
  // all-zero block, whose products are zero anyway); v * 2^-s is exact
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
  uint32_t o[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float v[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[4 * g + q]));
      v[2 * q] = f.x * inv;
      v[2 * q + 1] = f.y * inv;
    }
    o[g] = e2m1x8_from_f32(v);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One thread per 32-value block.  Threads are laid out by rows: a row is
// shared by tpr = 2^log2_tpr threads (the CTA takes kMxThreads / tpr rows
// at once) and thread i of a row quantizes its blocks i, i + tpr, ...; tpr
// is the smallest power of two that covers the row's blocks, up to the
// whole CTA.  A warp's 16-byte loads then cover whole 64-byte blocks of
// consecutive memory, and its stores of codes (16 bytes a thread) and of
// scale bytes are contiguous.  Measured on GB300 at 4096 x 4096: 8.8 us,
// against 13.0 us with four threads per block (a 16-byte load each and a
// 4-lane maximum): one thread per block also drops the shuffles and does
// the scale arithmetic once per block, not four times.  `vec_in` / `vec_out`:
// rows of X / of the codes start on 16-byte boundaries, so whole blocks
// move as 16-byte accesses; other layouts take element accesses.
constexpr int kQuantCtasPerSm = 4;

__global__ void __launch_bounds__(kMxThreads, kQuantCtasPerSm)
    quantize_mxf4_kernel(const __half* __restrict__ X, int64_t ldx, int64_t K, int64_t nblk,
                         int64_t rows, int log2_tpr, bool vec_in, bool vec_out,
                         uint8_t* __restrict__ codes, int64_t ldq_bytes,
                         uint8_t* __restrict__ scales, int64_t lds) {
  // Launched as a programmatic dependent: the grid is scheduled while the
  // kernel before it drains, and reads nothing before that kernel is done.
  // The GEMM that follows may be scheduled at once: it waits for this grid
  // to finish before reading the codes (and every CTA of this grid is
  // resident from the start: one wave).
  grid_dependency_wait();
  grid_launch_dependents();
  const int tpr = 1 << log2_tpr;
  const int in_row = threadIdx.x & (tpr - 1);
  const int rows_per_cta = kMxThreads >> log2_tpr;
  const int64_t row_step = static_cast<int64_t>(gridDim.x) * rows_per_cta;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * rows_per_cta + (threadIdx.x >> log2_tpr);
       r < rows; r += row_step) {
    const __half* xrow = X + r * ldx;
    uint8_t* qrow = codes + r * ldq_bytes;
    for (int64_t b = in_row; b < nblk; b += tpr) {
      const int64_t k0 = b * kMxBlock;
      const bool full = k0 + kMxBlock <= K;
      uint32_t w[16];
      if (full && vec_in) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = ld_nc16(xrow + k0 + 8 * q);
          w[4 * q] = v.x;
          w[4 * q + 1] = v.y;
          w[4 * q + 2] = v.z;
          w[4 * q + 3] = v.w;
        }
      } else {
        // element loads, zeros past K
        const uint16_t* s16 = reinterpret_cast<const uint16_t*>(xrow + k0);
        const int n = full ? kMxBlock : static_cast<int>(K - k0);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const uint32_t lo = 2 * q < n ? s16[2 * q] : 0u;
          const uint32_t hi = 2 * q + 1 < n ? s16[2 * q + 1] : 0u;
          w[q] = lo | (hi << 16);
        }
      }
      uint32_t scale_byte;
      const uint4 packed = quantize_block(w, scale_byte);
      uint8_t* dst = qrow + k0 / 2;
      if (full && vec_out) {
        *reinterpret_cast<uint4*>(dst) = packed;
      } else {
        // the block's bytes up to K (an odd K leaves the last high nibble 0)
        const int nbytes = full ? kMxBlock / 2 : static_cast<int>((K - k0 + 1) / 2);
        const uint32_t pw[4] = {packed.x, packed.y, packed.z, packed.w};
#pragma unroll
        for (int i = 0; i < kMxBlock / 2; ++i)
          if (i < nbytes) dst[i] = static_cast<uint8_t>(pw[i >> 2] >> (8 * (i & 3)));
      }
      scales[r * lds + b] = static_cast<uint8_t>(scale_byte);
    }
  }
}

// ---------------------------------------------------------------------------
// Widening to BF16
// ---------------------------------------------------------------------------

// One byte of two E2M1 codes -> two FP16 values (low nibble in the low half).
__device__ __forceinline__ __half2 e2m1x2_to_half2(uint32_t byte) {
  uint32_t o;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
      : "=r"(o)
      : "r"(byte));
  return *reinterpret_cast<__half2*>(&o);
}

// FP32 value of an E8M0 scale byte: 2^(e - 127); e = 0 is the FP32
// subnormal 2^-127; e = 255 is NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
  const uint32_t bits = e == 0 ? 0x00400000u : (e == 255 ? 0x7FC00000u : e << 23);
  return __uint_as_float(bits);
}

struct MxOperand {
  const uint8_t* codes;
  int64_t ld_bytes;  // row pitch of the codes (a multiple of 16)
  const uint8_t* scales;
  int64_t lds;       // row pitch of the scales
  int64_t units;     // rows * nblk: blocks of 32 values
  uint16_t* dst;     // BF16 rows of nblk * 32 values
  int dense;         // ld_bytes == 16 * nblk and lds == nblk: unit u at codes + 16 u, scales + u
};

// A unit (one block of one row: 16 bytes of codes and a scale byte in, 32
// BF16 values = 64 bytes out) is taken by 4 consecutive threads, each
// turning 4 code bytes into 16 output bytes: a warp reads 128 contiguous
// bytes of codes and writes 512 contiguous bytes.  Quarter-units of the
// first operand, then of the second; each thread issues kWidenUnroll loads
// before converting.
constexpr int kWidenUnroll = 4;

__device__ __forceinline__ const uint8_t* unit_codes(const MxOperand& op, int64_t u, int64_t nblk,
                                                     const uint8_t** scale) {
  if (op.dense) {
    *scale = op.scales + u;
    return op.codes + u * 16;
  }
  const int64_t r = u / nblk, b = u - r * nblk;
  *scale = op.scales + r * op.lds + b;
  return op.codes + r * op.ld_bytes + b * 16;
}

__global__ void __launch_bounds__(kMxThreads)
    widen_mxf4_kernel(MxOperand op0, MxOperand op1, int64_t nblk) {
  const int64_t total = 4 * (op0.units + op1.units);  // quarter-units
  const int64_t q0 = 4 * op0.units;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kMxThreads;
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * kMxThreads + threadIdx.x; i0 < total;
       i0 += stride * kWidenUnroll) {
    uint32_t w[kWidenUnroll], sc[kWidenUnroll];
#pragma unroll
    for (int t = 0; t < kWidenUnroll; ++t) {
      const int64_t i = i0 + t * stride;
      if (i < total) {
        const bool first = i < q0;
        const int64_t qi = first ? i : i - q0;
        const uint8_t* sp;
        const uint8_t* cp = unit_codes(first ? op0 : op1, qi >> 2, nblk, &sp);
        w[t] = __ldg(reinterpret_cast<const unsigned int*>(cp) + (qi & 3));
        sc[t] = *sp;
      }
    }
#pragma unroll
    for (int t = 0; t < kWidenUnroll; ++t) {
      const int64_t i = i0 + t * stride;
      if (i < total) {
        const bool first = i < q0;
        const int64_t qi = first ? i : i - q0;
        const float x = e8m0_to_f32(sc[t]);
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __half22float2(e2m1x2_to_half2((w[t] >> (8 * j)) & 0xFFu));
          const __nv_bfloat162 h = __floats2bfloat162_rn(f.x * x, f.y * x);
          o[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        // quarter qi: output values 8 qi .. 8 qi + 7 of the operand's copy
        *reinterpret_cast<uint4*>((first ? op0.dst : op1.dst) + qi * 8) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  // The GEMM launched next may be scheduled once every thread has issued its
  // copies (it waits for their completion before reading them).
  grid_launch_dependents();
}

int grid_for_units(int64_t units_per_thread_step, int sm_count) {
  const int64_t cap = static_cast<int64_t>(sm_count) * 8 * 4;
  const int64_t blocks = units_per_thread_step < cap ? units_per_thread_step : cap;
  return static_cast<int>(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_quantize_mxf4(int64_t rows, int64_t K, const void* X, int64_t ldx,
                                 void* codes, int64_t ldq, void* scales, int64_t lds,
                                 cudaStream_t stream, int sm_count) {
  const int64_t nblk = (K + kMxBlock - 1) / kMxBlock;
  if (rows <= 0 || nblk <= 0) return cudaSuccess;
  // threads per row: one per block, rounded up to a power of two, at most
  // the whole CTA
  int log2_tpr = 0;
  while (log2_tpr < 8 && (int64_t(1) << log2_tpr) < nblk) ++log2_tpr;
  const int64_t rows_per_cta = kMxThreads >> log2_tpr;
  const int64_t ctas = (rows + rows_per_cta - 1) / rows_per_cta;
  const int64_t cap = static_cast<int64_t>(sm_count) * kQuantCtasPerSm;  // one wave
  const int grid = static_cast<int>(ctas < cap ? ctas : cap);
  const bool vec_in = (reinterpret_cast<uintptr_t>(X) & 15) == 0 && ldx % 8 == 0;
  const bool vec_out = (reinterpret_cast<uintptr_t>(codes) & 15) == 0 && (ldq / 2) % 16 == 0;
  const cudaError_t e = launch_dependent(
      quantize_mxf4_kernel, dim3(static_cast<unsigned>(grid)), dim3(kMxThreads), 0, stream,
      static_cast<const __half*>(X), ldx, K, nblk, rows, log2_tpr, vec_in, vec_out,
      static_cast<uint8_t*>(codes), ldq / 2, static_cast<uint8_t*>(scales), lds);
  count_launches(1);
  return e;
}

cudaError_t launch_widen_mxf4(const MxWidenJob* jobs, int njobs, int64_t K, cudaStream_t stream,
                              int sm_count) {
  if (njobs < 1 || njobs > 2) return cudaErrorInvalidValue;
  const int64_t nblk = (K + kMxBlock - 1) / kMxBlock;
  MxOperand ops[2] = {};
  for (int i = 0; i < njobs; ++i) {
    ops[i].codes = static_cast<const uint8_t*>(jobs[i].codes);
    ops[i].ld_bytes = jobs[i].ld / 2;
    ops[i].scales = static_cast<const uint8_t*>(jobs[i].scales);
    ops[i].lds = jobs[i].lds;
    ops[i].units = jobs[i].rows * nblk;
    ops[i].dst = reinterpret_cast<uint16_t*>(jobs[i].dst);
    ops[i].dense = ops[i].ld_bytes == 16 * nblk && ops[i].lds == nblk;
  }
  const int64_t total = 4 * (ops[0].units + ops[1].units);
  if (total <= 0) return cudaSuccess;
  const int grid =
      grid_for_units((total + kMxThreads * kWidenUnroll - 1) / (kMxThreads * kWidenUnroll),
                     sm_count);
  widen_mxf4_kernel<<<grid, kMxThreads, 0, stream>>>(ops[0], ops[1], nblk);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dg
