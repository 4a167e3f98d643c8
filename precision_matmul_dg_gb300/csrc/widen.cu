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

#include <type_traits>

#include "convert.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dg {
namespace {

// The copy is written in chunks of 16 bytes (8 FP16 values), each made from
// 8 int8 bytes or 4 bytes of packed E2M1 codes.  Consecutive threads take
// consecutive chunks, so a warp reads one contiguous run of 256 or 128 bytes
// and writes 512 contiguous bytes.  Each thread issues kUnroll loads before
// its first conversion.  Whole 16-byte source groups are read up to the row
// pitch (a multiple of 16 bytes); columns >= K of the copy are never read by
// the GEMM.
constexpr int kWidenThreads = 256;
constexpr int kUnroll = 4;

template <bool kE2M1>
struct WidenChunk {
  static constexpr int kInBytes = kE2M1 ? 4 : 8;   // source bytes per chunk
  static constexpr int kPerGroup = 16 / kInBytes;  // chunks per 16-byte source group
  using In = typename std::conditional<kE2M1, uint32_t, uint2>::type;
  static __device__ __forceinline__ In load(const uint8_t* p) {
    if constexpr (kE2M1)
      return ld_stream4(p);
    else
      return ld_stream8(p);
  }
  static __device__ __forceinline__ uint4 convert(const In& w) {
    if constexpr (kE2M1) {
      return e2m1x8_to_f16x8(w);
    } else {
      return make_uint4(i8x2_to_f16x2(w.x & 0xFFFFu), i8x2_to_f16x2(w.x >> 16),
                        i8x2_to_f16x2(w.y & 0xFFFFu), i8x2_to_f16x2(w.y >> 16));
    }
  }
};

// Rows packed back to back in both source and copy (the usual case): an
// operand is one run of chunks.  One launch widens up to two operands (A and
// B of an INT8 product): chunks [0, total0) of the first, then total1 of the
// second, taken kUnroll per thread step.
template <bool kE2M1>
__global__ void __launch_bounds__(kWidenThreads)
    widen_dense_kernel(const uint8_t* __restrict__ src0, __half* __restrict__ dst0, int64_t total0,
                       const uint8_t* __restrict__ src1, __half* __restrict__ dst1,
                       int64_t total1) {
  using C = WidenChunk<kE2M1>;
  const int64_t total = total0 + total1;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWidenThreads;
  for (int64_t i0 = blockIdx.x * static_cast<int64_t>(kWidenThreads) + threadIdx.x; i0 < total;
       i0 += stride * kUnroll) {
    typename C::In w[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < total)
        w[u] = C::load(i < total0 ? src0 + i * C::kInBytes : src1 + (i - total0) * C::kInBytes);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < total)
        *reinterpret_cast<uint4*>(i < total0 ? dst0 + i * 8 : dst1 + (i - total0) * 8) =
            C::convert(w[u]);
    }
  }
  // The GEMM launched next (a programmatic dependent) may be scheduled once
  // every thread has issued its copies; it waits for their completion.
  grid_launch_dependents();
}

// Padded rows: a block takes rows blockIdx.x, blockIdx.x + gridDim.x, ...;
// in a row its threads take chunks tx, tx + blockDim.x, ...
template <bool kE2M1>
__global__ void __launch_bounds__(kWidenThreads)
    widen_rows_kernel(const uint8_t* __restrict__ src, int rows, int groups,
                      int64_t ld_src_bytes, __half* __restrict__ dst, int64_t ld_dst) {
  using C = WidenChunk<kE2M1>;
  const int chunks = groups * C::kPerGroup;
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint8_t* s = src + static_cast<int64_t>(r) * ld_src_bytes;
    __half* d = dst + static_cast<int64_t>(r) * ld_dst;
    for (int c0 = threadIdx.x; c0 < chunks; c0 += kWidenThreads * kUnroll) {
      typename C::In w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + u * kWidenThreads;
        if (c < chunks) w[u] = C::load(s + static_cast<int64_t>(c) * C::kInBytes);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + u * kWidenThreads;
        if (c < chunks)
          *reinterpret_cast<uint4*>(d + static_cast<int64_t>(c) * 8) = C::convert(w[u]);
      }
    }
  }
  // The GEMM launched next (a programmatic dependent) may be scheduled once
  // every thread has issued its copies; it waits for their completion.
  grid_launch_dependents();
}

// Blocks: enough for `items` work items per thread step, capped at four
// waves of eight resident blocks per SM.
int grid_for(int64_t items, int sm_count) {
  const int64_t cap = static_cast<int64_t>(sm_count) * 8 * 4;
  const int64_t blocks = items < cap ? items : cap;
  return static_cast<int>(blocks < 1 ? 1 : blocks);
}

}  // namespace

int64_t widened_ld(int64_t K) { return (K + 31) / 32 * 32; }

namespace {

struct WidenShape {
  int64_t groups, pitch, out_per_group;
  bool dense;
};

WidenShape widen_shape(const WidenJob& j, int64_t K) {
  const bool e2m1 = j.dtype == DG_E2M1;
  WidenShape w;
  // 16-byte source groups per row: 16 int8 or 32 E2M1 codes; the source row
  // pitch (ld_src bytes, or ld_src / 2 for E2M1) is a multiple of 16
  w.groups = e2m1 ? ((K + 1) / 2 + 15) / 16 : (K + 15) / 16;
  w.pitch = e2m1 ? j.ld_src / 2 : j.ld_src;
  w.out_per_group = e2m1 ? 32 : 16;
  w.dense = w.pitch == w.groups * 16 && widened_ld(K) == w.groups * w.out_per_group;
  return w;
}

cudaError_t launch_rows(const WidenJob& j, const WidenShape& w, int64_t K, cudaStream_t stream,
                        int sm_count) {
  if (j.rows > INT32_MAX || w.groups > INT32_MAX) return cudaErrorInvalidValue;
  const int grid = grid_for(j.rows, sm_count);
  const auto* s = static_cast<const uint8_t*>(j.src);
  // An ordinary launch (see widen_dense_kernel)
  (j.dtype == DG_E2M1 ? widen_rows_kernel<true> : widen_rows_kernel<false>)
      <<<grid, kWidenThreads, 0, stream>>>(s, static_cast<int>(j.rows), static_cast<int>(w.groups),
                                           w.pitch, j.dst, widened_ld(K));
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_widen(const WidenJob* jobs, int njobs, int64_t K, cudaStream_t stream,
                         int sm_count) {
  if (njobs < 1 || njobs > 2) return cudaErrorInvalidValue;
  for (int i = 0; i < njobs; ++i)
    if (jobs[i].dtype != DG_I8 && jobs[i].dtype != DG_E2M1) return cudaErrorInvalidValue;
  const WidenShape w0 = widen_shape(jobs[0], K);
  const WidenShape w1 = njobs == 2 ? widen_shape(jobs[1], K) : WidenShape{0, 0, 0, true};
  const bool fused = w0.dense && w1.dense && (njobs == 1 || jobs[1].dtype == jobs[0].dtype);
  if (!fused) {
    for (int i = 0; i < njobs; ++i) {
      const WidenShape& w = i == 0 ? w0 : w1;
      cudaError_t e;
      if (w.dense) {
        const WidenJob one[1] = {jobs[i]};
        e = launch_widen(one, 1, K, stream, sm_count);
      } else {
        e = launch_rows(jobs[i], w, K, stream, sm_count);
      }
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  // chunks of 16 output bytes: 2 per source group of int8, 4 of E2M1
  const int64_t per_group = jobs[0].dtype == DG_E2M1 ? 4 : 2;
  const int64_t t0 = jobs[0].rows * w0.groups * per_group;
  const int64_t t1 = njobs == 2 ? jobs[1].rows * w1.groups * per_group : 0;
  const auto* s0 = static_cast<const uint8_t*>(jobs[0].src);
  const auto* s1 = njobs == 2 ? static_cast<const uint8_t*>(jobs[1].src) : s0;
  __half* d1 = njobs == 2 ? jobs[1].dst : jobs[0].dst;
  const int grid =
      grid_for((t0 + t1 + kWidenThreads * kUnroll - 1) / (kWidenThreads * kUnroll), sm_count);
  // An ordinary launch: as a programmatic dependent, its small blocks would
  // wait beside the previous GEMM's CTAs through their last epilogue and slow
  // it (measured: 6 us on a 2048 x 8960 x 1536 bias+GELU GEMM).
  (jobs[0].dtype == DG_E2M1 ? widen_dense_kernel<true> : widen_dense_kernel<false>)
      <<<grid, kWidenThreads, 0, stream>>>(s0, jobs[0].dst, t0, s1, d1, t1);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dg
