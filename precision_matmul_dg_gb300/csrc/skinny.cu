// Skinny W4A16 GEMM: D = epilogue(alpha * A . B + beta * C) for M <= 16 rows
// of FP16 activations A against packed 4-bit E2M1 weights B (N rows of K
// codes, two per byte, k = 2p in the low nibble of byte p; discosf.com/news/
// 5532976, section 4.3 packing and section 3.2's W4A16 shapes with M = 16).
//
// At M <= 16 the product reads each weight once and does 16 multiply-adds
// with it: the job is streaming N*K/2 bytes of weights from HBM.  The CUDA
// cores cannot keep up (16 FMAs per 4-bit weight), and staging widened weight
// tiles in shared memory for tcgen05 costs more than the MMA saves at this
// size.  So the weights go from HBM straight into registers, are widened
// there with cvt.rn.f16x2.e2m1x2 and fed to warp-level m16n8k16 MMAs (FP16 in,
// FP32 accumulate), with the 16 activation rows (zero-padded) in shared memory.
//
// Layout.  A block of 16 warps owns 64 columns: warp w takes column group
// w % 8 (8 columns, one B row per group of 4 lanes) and K half w / 8 (every
// other pair of 128-code windows).  A warp reads a window pair of its 8 rows
// (8 x 128 bytes) with two loads of 4 whole 128-byte lines each, all of its
// pairs of a 2048-code chunk before the first MMA, then shuffles the bytes so
// that lane (grp = lane / 4, tig = lane % 4) holds, per window, the 16 bytes
// (32 codes) at window offset 32 * tig of B row n0 + grp (whole-line loads
// take half the memory requests of per-lane 16-byte pieces of 8 rows).
// For MMA step s (0..7) of a window it uses bytes 2s and 2s + 1 of those 16:
// codes 4s .. 4s + 3, which fill the B fragment slots k = 2 tig, 2 tig + 1
// and 2 tig + 8, 2 tig + 9.  The A fragment takes the same four K positions
// of rows grp and grp + 8 from shared memory, so every MMA step covers 16
// distinct K values of the window and the K order inside the dot product is
// merely permuted.  The activation chunk is staged in shared memory twice:
// row-major as loaded (16-byte stores), then rearranged once into fragment
// order (window, step, lane: the lane's four 32-bit A registers side by
// side), so that in the MMA loop a step's A fragment is one conflict-free
// 16-byte load.  Read row-major, every step cost two 8-byte loads at a
// 4-way bank conflict, and the eight column-group warps each read all of A.
// The two K halves are summed in shared memory; the fused
// epilogue (alpha, beta * C, bias, erf-GELU, FP16 rounding) runs on the MMA
// fragments.  Columns >= N and rows >= M are computed on clamped or zero
// inputs and never stored; codes at k >= K meet zeroed activations.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "convert.cuh"
#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dg {
namespace {

constexpr int kSkWarps = 16;     // 8 column groups x 2 K halves
constexpr int kSkThreads = kSkWarps * 32;
constexpr int kSkGroups = 8;     // column groups of 8 per block
constexpr int kSkCols = kSkGroups * 8;
constexpr int kSkWindow = 128;   // codes per window: 16 bytes per lane
constexpr int kSkBatch = 8;      // windows per warp per chunk (all loads in flight)
constexpr int kSkPairs = kSkBatch / 2;  // window pairs per warp per chunk
constexpr int kSkChunk = 2 * kSkBatch * kSkWindow;  // K codes per activation chunk
// activations of a chunk in fragment order: [window][step][lane] x 16 bytes
constexpr int kSkSmemA = (kSkChunk / kSkWindow) * 8 * 32 * 16;
static_assert(kSkSmemA == 16 * kSkChunk * 2, "16 rows of a chunk");
// and row-major as loaded, rows padded by 16 bytes
constexpr int kSkRowStride = kSkChunk + 8;  // halves
constexpr int kSkSmemRows = 16 * kSkRowStride * 2;
constexpr int kSkAPer = 16 * (kSkChunk / 8) / kSkThreads;  // 16-byte pieces per thread
static_assert(kSkAPer * kSkThreads == 16 * (kSkChunk / 8), "whole pieces per thread");
constexpr int kSkSmemRed = kSkGroups * 32 * 4 * 4;
constexpr int kSkSmem = kSkSmemA + kSkSmemRows + kSkSmemRed;

struct SkParams {
  int M, N, K;
  const __half* A;
  int64_t lda;
  const uint8_t* B;
  int64_t ldb_bytes;  // packed row pitch
  const __half* C;    // read when beta != 0
  int64_t ldc;
  __half* D;
  int64_t ldd;
  const __half* bias;
  Epi epi;
};
static_assert(sizeof(SkParams) <= 128, "parameter struct within 128 bytes (see Epi)");

// d += a (16 x 16, row-major fragment) . b (16 x 8, column-major fragment)
__device__ __forceinline__ void mma_m16n8k16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kSkThreads)
    skinny_w4a16_kernel(const SkParams p, const __grid_constant__ EpiProgram prog) {
  extern __shared__ __align__(16) uint8_t sk_smem[];
  uint32_t* As = reinterpret_cast<uint32_t*>(sk_smem);  // [window][step][lane][4]
  __half* Ar = reinterpret_cast<__half*>(sk_smem + kSkSmemA);  // [16][kSkRowStride]
  float* red = reinterpret_cast<float*>(sk_smem + kSkSmemA + kSkSmemRows);  // [8][32][4]
  grid_dependency_wait();  // launched as a dependent of the previous kernel

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cg = warp % kSkGroups, kh = warp / kSkGroups;
  const int grp = lane >> 2, tig = lane & 3;
  const int n0 = blockIdx.x * kSkCols + cg * 8;
  // this lane's rows for the line loads: n0 + lane / 8 and n0 + 4 + lane / 8
  // (rows >= N: clamped, results not stored)
  const uint8_t* brow0 = p.B + static_cast<int64_t>(min(n0 + (lane >> 3), p.N - 1)) * p.ldb_bytes;
  const uint8_t* brow1 =
      p.B + static_cast<int64_t>(min(n0 + 4 + (lane >> 3), p.N - 1)) * p.ldb_bytes;
  const int row_groups = (p.K + 31) / 32;  // 16-byte groups holding codes < K
  // The epilogue's inputs of this lane (warps of the first K half: bias of
  // columns n0 + 2 tig + {0, 1}, C at rows grp and grp + 8), loaded now so
  // that they arrive while the weights stream.
  float pre_b[2] = {0.0f, 0.0f}, pre_c[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};
  if (kh == 0) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int nn = n0 + 2 * tig + e;
      if (nn >= p.N) continue;
      if (p.epi.flags & kEpiBias) pre_b[e] = __half2float(p.bias[nn]);
      if (p.epi.beta != 0.0f) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int m = grp + 8 * h;
          if (m < p.M) pre_c[h][e] = __half2float(p.C[static_cast<int64_t>(m) * p.ldc + nn]);
        }
      }
    }
  }
  // Two independent accumulator chains (even and odd MMA steps): one chain
  // of dependent MMAs per warp would be bound by the MMA latency.
  float acc2[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};

  for (int kc0 = 0; kc0 < p.K; kc0 += kSkChunk) {
    const int nwin = (min(kSkChunk, p.K - kc0) + kSkWindow - 1) / kSkWindow;
    // this warp's weight loads for the chunk, issued before anything waits:
    // window pair q = kh + 2i covers bytes [128 q, 128 q + 128) of each row
    uint4 bl[kSkPairs][2];
#pragma unroll
    for (int i = 0; i < kSkPairs; ++i) {
      const int q = kh + 2 * i;
      const int g = kc0 / 32 + q * 8 + (lane & 7);
      const bool in = 2 * q < nwin && g < row_groups;
      bl[i][0] = in ? ld_stream16(brow0 + static_cast<int64_t>(g) * 16) : make_uint4(0u, 0u, 0u, 0u);
      bl[i][1] = in ? ld_stream16(brow1 + static_cast<int64_t>(g) * 16) : make_uint4(0u, 0u, 0u, 0u);
    }
    // activation chunk -> shared memory; rows >= M and columns >= K are zero.
    // A thread's kSkAPer 16-byte pieces are all loaded before any is stored,
    // so the chunk costs one round trip to L2 rather than one per piece.
    __syncthreads();  // the previous chunk's reads are done
    {
      uint4 v[kSkAPer];
#pragma unroll
      for (int i = 0; i < kSkAPer; ++i) {
        const int idx = threadIdx.x + i * kSkThreads;
        const int r = idx / (kSkChunk / 8), u = idx % (kSkChunk / 8);
        const int k = kc0 + u * 8;
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (r < p.M && k < p.K)
          v[i] = __ldg(reinterpret_cast<const uint4*>(p.A + static_cast<int64_t>(r) * p.lda + k));
      }
#pragma unroll
      for (int i = 0; i < kSkAPer; ++i) {
        const int idx = threadIdx.x + i * kSkThreads;
        const int r = idx / (kSkChunk / 8), u = idx % (kSkChunk / 8);
        const int k = kc0 + u * 8;
        if (k < p.K && k + 8 > p.K) {
          __half* h = reinterpret_cast<__half*>(&v[i]);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (k + e >= p.K) h[e] = __ushort_as_half(0);
        }
        *reinterpret_cast<uint4*>(Ar + r * kSkRowStride + u * 8) = v[i];
      }
    }
    __syncthreads();
    // fragment slot q = (window w, step s, lane (grp, tig)): rows grp and
    // grp + 8 at window offset 32 tig + 4s .. + 3, as the registers
    // {row grp (+0, +1), row grp + 8 (+0, +1), row grp (+2, +3), row grp + 8 (+2, +3)}
#pragma unroll
    for (int i = 0; i < (kSkSmemA / 16) / kSkThreads; ++i) {
      const int q = threadIdx.x + i * kSkThreads;
      const int ln = q & 31, st = (q >> 5) & 7, w = q >> 8;
      const int k = w * kSkWindow + 32 * (ln & 3) + 4 * st;
      const uint2 lo = *reinterpret_cast<const uint2*>(Ar + (ln >> 2) * kSkRowStride + k);
      const uint2 hi = *reinterpret_cast<const uint2*>(Ar + ((ln >> 2) + 8) * kSkRowStride + k);
      reinterpret_cast<uint4*>(As)[q] = make_uint4(lo.x, hi.x, lo.y, hi.y);
    }
    __syncthreads();
    // lane (grp, tig) takes, for window h of a pair, piece 4h + tig of row
    // grp, held by lane 8 (grp % 4) + 4h + tig of load grp / 4
#pragma unroll
    for (int i = 0; i < kSkBatch; ++i) {
      const int w = 2 * (kh + 2 * (i >> 1)) + (i & 1);
      if (w >= nwin) break;  // the same for the whole warp
      const int src = 8 * (grp & 3) + 4 * (i & 1) + tig;
      const uint4 v0 = bl[i >> 1][0], v1 = bl[i >> 1][1];
      // every lane takes part in both shuffles, then keeps the one for its row
      const uint32_t s0[4] = {__shfl_sync(0xffffffffu, v0.x, src), __shfl_sync(0xffffffffu, v0.y, src),
                              __shfl_sync(0xffffffffu, v0.z, src), __shfl_sync(0xffffffffu, v0.w, src)};
      const uint32_t s1[4] = {__shfl_sync(0xffffffffu, v1.x, src), __shfl_sync(0xffffffffu, v1.y, src),
                              __shfl_sync(0xffffffffu, v1.z, src), __shfl_sync(0xffffffffu, v1.w, src)};
      uint32_t wv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) wv[j] = grp < 4 ? s0[j] : s1[j];
      const uint4* af = reinterpret_cast<const uint4*>(As) + w * 8 * 32 + lane;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // word j: codes 8j .. 8j + 7 of the lane's 32, bytes 2s and 2s + 1
        // for steps s = 2j and 2j + 1
        uint32_t bf[4];
        e2m1x8_to_f16x2x4(wv[j], bf);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int s = 2 * j + h;
          // rows grp and grp + 8 at the step's K positions 32 tig + 4s .. + 3
          const uint4 f = af[s * 32];
          const uint32_t a[4] = {f.x, f.y, f.z, f.w};
          mma_m16n8k16(acc2[h], a, bf[2 * h], bf[2 * h + 1]);  // codes 4s .. 4s + 3
        }
      }
    }
  }

  float acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = acc2[0][j] + acc2[1][j];
  // the two K halves of each column group
  if (kh == 1) {
#pragma unroll
    for (int j = 0; j < 4; ++j) red[(cg * 32 + lane) * 4 + j] = acc[j];
  }
  __syncthreads();
  grid_launch_dependents();  // the weights have been streamed
  if (kh != 0) return;
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] += red[(cg * 32 + lane) * 4 + j];
  // fragment: acc[0..1] at (row grp, columns n0 + 2 tig + {0,1}), acc[2..3] at row grp + 8
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int m = grp + 8 * h;
    if (m >= p.M) continue;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int nn = n0 + 2 * tig + e;
      if (nn >= p.N) continue;
      const float t = epi_apply(acc[2 * h + e], pre_c[h][e], pre_b[e], p.epi, prog);
      epi_store(p.D, static_cast<int64_t>(m) * p.ldd + nn, t, p.epi, prog);
    }
  }
}

}  // namespace

int skinny_smem_bytes() { return kSkSmem; }
int skinny_threads() { return kSkThreads; }
int skinny_cols_per_block() { return kSkCols; }
int skinny_k_chunk() { return kSkChunk; }
int skinny_kernel_regs() {
  static std::atomic<int> slot{-1};
  return kernel_regs(skinny_w4a16_kernel, slot);
}

cudaError_t launch_skinny(const GemmArgs& a, const dg_tile_plan& plan) {
  (void)plan;
  if (a.M > 16 || a.dtype_a != DG_F16 || a.dtype_b != DG_E2M1) return cudaErrorInvalidValue;
  SkParams p;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.A = static_cast<const __half*>(a.A);
  p.lda = a.lda;
  p.B = static_cast<const uint8_t*>(a.B);
  p.ldb_bytes = a.ldb / 2;
  p.C = static_cast<const __half*>(a.C);
  p.ldc = a.ldc;
  p.D = static_cast<__half*>(a.D);
  p.ldd = a.ldd;
  p.bias = static_cast<const __half*>(a.bias);
  p.epi = make_epi(a);
  int dev = 0;
  cudaGetDevice(&dev);
  static std::atomic<uint64_t> attr_set{0};  // one shared-memory opt-in per device
  const cudaError_t ea = once_per_device(attr_set, dev, []() {
    return cudaFuncSetAttribute(skinny_w4a16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSkSmem);
  });
  if (ea != cudaSuccess) return ea;
  const unsigned grid = static_cast<unsigned>((a.N + kSkCols - 1) / kSkCols);
  const cudaError_t e = launch_dependent(skinny_w4a16_kernel, dim3(grid), dim3(kSkThreads),
                                         kSkSmem, a.stream, p, make_program(a));
  count_launches(1);
  return e;
}

}  // namespace dg
