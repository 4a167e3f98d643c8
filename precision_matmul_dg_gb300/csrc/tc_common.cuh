// Pieces shared by the tensor-core GEMM kernels: tile order, the fused FP16
// epilogue of one 32-column accumulator chunk, and tensor-map construction.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dg {
namespace tc {

constexpr int kBlockM = 128;  // accumulator rows per CTA (TMEM lanes)
constexpr int kBlockK = 64;   // K elements per pipeline stage (128 bytes of FP16)

// Grouped tile order: `group_m` row blocks are walked together so that
// concurrently running CTAs share A and B panels in L2.
__device__ __forceinline__ void tile_coords(int t, int num_m_blocks, int num_n_blocks,
                                            int group_m, int& m_blk, int& n_blk) {
  const int per_group = group_m * num_n_blocks;
  const int g = t / per_group;
  const int first_m = g * group_m;
  const int gm = min(num_m_blocks - first_m, group_m);
  const int r = t - g * per_group;
  m_blk = first_m + r % gm;
  n_blk = r / gm;
}

// Fused FP16 epilogue for one thread's row and 32 consecutive columns:
// D = round_fp16(GELU?(alpha*acc + beta*C + bias)).  C and D share `cd`
// (leading dimension N).  Rows >= M and columns >= N are skipped.
__device__ __forceinline__ void epilogue_f16_chunk(const uint32_t (&r)[32], int row, int col0,
                                                   int M, int N, const Epi& epi, __half* cd,
                                                   const __half* bias) {
  if (row >= M) return;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = epi.alpha * __uint_as_float(r[i]);
  __half* drow = cd + static_cast<int64_t>(row) * N;
  const bool full = (col0 + 32 <= N) && ((N & 7) == 0);
  if (epi.beta != 0.0f) {
    if (full) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 cv = *reinterpret_cast<const uint4*>(drow + col0 + q * 8);
        const __half2* ch = reinterpret_cast<const __half2*>(&cv);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float2 f = __half22float2(ch[h]);
          v[q * 8 + 2 * h] = fmaf(epi.beta, f.x, v[q * 8 + 2 * h]);
          v[q * 8 + 2 * h + 1] = fmaf(epi.beta, f.y, v[q * 8 + 2 * h + 1]);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (col0 + i < N) v[i] = fmaf(epi.beta, __half2float(drow[col0 + i]), v[i]);
    }
  }
  if (epi.flags & kEpiBias) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col0 + i < N) v[i] += __half2float(__ldg(bias + col0 + i));
  }
  if (epi.flags & kEpiGelu) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = gelu_erf(v[i]);
  }
  if (full) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 ov;
      __half2* oh = reinterpret_cast<__half2*>(&ov);
#pragma unroll
      for (int h = 0; h < 4; ++h) oh[h] = __floats2half2_rn(v[q * 8 + 2 * h], v[q * 8 + 2 * h + 1]);
      *reinterpret_cast<uint4*>(drow + col0 + q * 8) = ov;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col0 + i < N) drow[col0 + i] = __float2half_rn(v[i]);
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// 2-D tensor map over `rows` rows of `inner` elements (row pitch `pitch_bytes`),
// box of box_rows x box_inner elements, zero fill outside the tensor.
// Encoded maps are kept in a small per-thread cache keyed by every argument
// (a map holds only an address and a layout, so a hit is always valid).
inline cudaError_t make_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                               int64_t rows, int64_t inner, int64_t pitch_bytes, int box_rows,
                               int box_inner, CUtensorMapSwizzle swizzle) {
  struct Entry {
    const void* base;
    int64_t rows, inner, pitch;
    int box_rows, box_inner, dtype, swizzle;
    CUtensorMap map;
  };
  constexpr int kCache = 16;
  thread_local Entry cache[kCache];
  thread_local int used = 0, next = 0;
  for (int i = 0; i < used; ++i) {
    const Entry& c = cache[i];
    if (c.base == base && c.rows == rows && c.inner == inner && c.pitch == pitch_bytes &&
        c.box_rows == box_rows && c.box_inner == box_inner && c.dtype == static_cast<int>(dtype) &&
        c.swizzle == static_cast<int>(swizzle)) {
      *map = c.map;
      return cudaSuccess;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner),
                             static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  Entry& e = cache[next];
  e.base = base;
  e.rows = rows;
  e.inner = inner;
  e.pitch = pitch_bytes;
  e.box_rows = box_rows;
  e.box_inner = box_inner;
  e.dtype = static_cast<int>(dtype);
  e.swizzle = static_cast<int>(swizzle);
  e.map = *map;
  next = (next + 1) % kCache;
  if (used < kCache) ++used;
  return cudaSuccess;
}

// K-major FP16 operand tile: box_rows x 64 elements, 128-byte swizzle.
inline cudaError_t make_f16_kmajor_map(CUtensorMap* map, const void* base, int64_t rows, int64_t k,
                                       int64_t ld, int box_rows) {
  return make_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, rows, k, ld * 2, box_rows,
                     kBlockK, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace tc
}  // namespace dg
