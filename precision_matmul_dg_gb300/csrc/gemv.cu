// Thin-M GEMM on the CUDA cores: y[m, j] = sum_k a[m, k] * B[j, k] for M <= 8.
//
// The "DeepGEMM" articles single out thin shapes that template libraries
// handle badly: M=1 with N=4096, K=131072 and M=1, N=256, K=12800
// (kwkr.cn/news/562171, section 2.1), and a small M=1 projection for which
// plain FMA beats the tensor cores (discosf.com/news/5532976, section 5.3,
// "use_hmma: false").  At M <= 8 the work is one pass over B, so this kernel
// is built for HBM bandwidth:
//   * one warp streams one row of B (one output column) over a K range with
//     128-bit non-allocating loads, several in flight per lane;
//   * each lane keeps FP32 partial sums in registers, then the warp reduces
//     them with xor-shuffles (discosf.com article, section 4.1 stage 3: warp
//     partial sums via shfl.sync rather than shared memory);
//   * long K is split over grid.y (split-K).  Each split writes FP32 partials
//     to a workspace; the last CTA of a row group to arrive adds the splits in
//     index order (deterministic) and applies the fused epilogue.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <algorithm>
#include <mutex>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dg {
namespace {

constexpr int kGemvWarps = 8;     // warps (= B rows) per CTA
constexpr int kGemvUnroll = 4;    // 16-byte loads in flight per lane per row
constexpr int kGemvMaxM = 8;

struct GemvParams {
  int M, N, K;
  const __half* A;
  int64_t lda;
  const __half* B;
  int64_t ldb;
  const __half* C;  // read when beta != 0
  int64_t ldc;
  __half* D;
  int64_t ldd;
  const __half* bias;
  Epi epi;
  int split_k;
  int k_chunk;  // K elements per split (multiple of 8)
  float* partial;       // [split_k][M][N] when split_k > 1
  unsigned* counters;   // [gridDim.x] when split_k > 1, zero between launches
};
static_assert(sizeof(GemvParams) <= 128, "parameter struct within 128 bytes (see Epi)");

// Strided batch: problem z (blockIdx.z) reads A + z sa, B + z sb, C + z sc
// and bias + z sbias and writes D + z sd (elements); its split-K partials
// and counters follow those of problem z - 1.
struct GemvBatch {
  int64_t sa, sb, sc, sd, sbias;
  const struct GemvGroupProblem* group;  // grouped launch: problem z is group[z] instead
};

// One problem of a grouped launch (dg_gemm_grouped): its rows and buffers
// (C and D one buffer of leading dimension N).  The launch's p.M is the
// largest M of the group, which sizes each problem's split-K partials.
struct GemvGroupProblem {
  const __half* A;
  const __half* B;
  __half* CD;
  const __half* bias;
  int64_t M;
};

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void fma8(float& acc, const uint4& a, const uint4& b) {
  const __half2* ah = reinterpret_cast<const __half2*>(&a);
  const __half2* bh = reinterpret_cast<const __half2*>(&b);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fa = __half22float2(ah[i]);
    const float2 fb = __half22float2(bh[i]);
    acc = fmaf(fa.x, fb.x, acc);
    acc = fmaf(fa.y, fb.y, acc);
  }
}

// sum over sp = 0 .. splits-1 of part[sp * stride], added in index order.
// The loads go out eight at a time (they do not depend on one another), so a
// reduction costs one L2 round trip per eight splits, not one per split.
__device__ __forceinline__ float sum_splits(const float* part, int64_t stride, int splits) {
  float s = 0.0f;
  int sp = 0;
  for (; sp + 8 <= splits; sp += 8) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __ldcg(part + (sp + i) * stride);
#pragma unroll
    for (int i = 0; i < 8; ++i) s += v[i];
  }
  for (; sp < splits; ++sp) s += __ldcg(part + sp * stride);
  return s;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One problem's output side: C, D and bias already offset to the problem.
struct GemvOut {
  const __half* C;
  __half* D;
  const __half* bias;
};

__device__ __forceinline__ void write_out(const GemvParams& p, const GemvOut& o,
                                          const EpiProgram& prog, int m, int j, float acc) {
  const float c = (p.epi.beta != 0.0f) ? __half2float(o.C[static_cast<int64_t>(m) * p.ldc + j])
                                        : 0.0f;
  const float b = (p.epi.flags & kEpiBias) ? __half2float(o.bias[j]) : 0.0f;
  epi_store(o.D, static_cast<int64_t>(m) * p.ldd + j, epi_apply(acc, c, b, p.epi, prog), p.epi,
            prog);
}

// This warp's partial dot products of B row j with the M rows of A over
// [k0, k1), one FP32 sum per lane and row (not yet reduced across the warp).
// Batches of `Unroll` 256-element steps: every load of a batch is in flight
// at once (one memory round trip per batch); steps past the end of the K
// range are predicated off.
template <int MROWS, int Unroll>
__device__ __forceinline__ void gemv_accumulate(const GemvParams& p, const __half* A,
                                                const __half* B, int j, int lane, int k0, int k1,
                                                float (&acc)[MROWS]) {
#pragma unroll
  for (int m = 0; m < MROWS; ++m) acc[m] = 0.0f;
  if (j >= p.N || k0 >= k1) return;
  const __half* brow = B + static_cast<int64_t>(j) * p.ldb;
  int k = k0 + lane * 8;
  constexpr int kStep = 256;
  // full batches: no predicates in the streaming loop
  for (; k + (Unroll - 1) * kStep + 8 <= k1; k += Unroll * kStep) {
    uint4 bv[Unroll];
#pragma unroll
    for (int u = 0; u < Unroll; ++u) bv[u] = ld_stream(brow + k + u * kStep);
#pragma unroll
    for (int u = 0; u < Unroll; ++u) {
#pragma unroll
      for (int m = 0; m < MROWS; ++m) {
        if (m < p.M) {
          const uint4 av = __ldg(reinterpret_cast<const uint4*>(
              A + static_cast<int64_t>(m) * p.lda + k + u * kStep));
          fma8(acc[m], av, bv[u]);
        }
      }
    }
  }
  // at most one partial batch, predicated per step
  if (k + 8 <= k1) {
    uint4 bv[Unroll];
#pragma unroll
    for (int u = 0; u < Unroll; ++u)
      bv[u] = (k + u * kStep + 8 <= k1) ? ld_stream(brow + k + u * kStep) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < Unroll; ++u) {
      if (k + u * kStep + 8 <= k1) {
#pragma unroll
        for (int m = 0; m < MROWS; ++m) {
          if (m < p.M) {
            const uint4 av = __ldg(reinterpret_cast<const uint4*>(
                A + static_cast<int64_t>(m) * p.lda + k + u * kStep));
            fma8(acc[m], av, bv[u]);
          }
        }
      }
    }
  }
  // k is now past the last whole 8-element group this lane owns; the ragged
  // tail (< 8 elements at the end of the K range) is done by the lane whose
  // next group would have started there.
  k = k1 - ((k1 - k0) & 7);
  if ((k - k0) % kStep == lane * 8 && k < k1) {
    for (int kk = k; kk < k1; ++kk) {
      const float bf = __half2float(brow[kk]);
#pragma unroll
      for (int m = 0; m < MROWS; ++m)
        if (m < p.M)
          acc[m] = fmaf(__half2float(A[static_cast<int64_t>(m) * p.lda + kk]), bf, acc[m]);
    }
  }
}

template <int MROWS>
__global__ void __launch_bounds__(kGemvWarps * 32)
    gemv_splitk_kernel(const GemvParams p, const __grid_constant__ EpiProgram prog,
                       const GemvBatch bt) {
  grid_dependency_wait();  // launched as a dependent of the previous kernel
  const int64_t z = blockIdx.z;
  const __half* A = p.A + z * bt.sa;
  const __half* B = p.B + z * bt.sb;
  const GemvOut out{p.C + z * bt.sc, p.D + z * bt.sd, p.bias ? p.bias + z * bt.sbias : nullptr};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.x * kGemvWarps + warp;
  const int split = blockIdx.y;
  const int k0 = split * p.k_chunk;
  const int k1 = min(p.K, k0 + p.k_chunk);

  float acc[MROWS];
  gemv_accumulate<MROWS, kGemvUnroll>(p, A, B, j, lane, k0, k1, acc);

#pragma unroll
  for (int m = 0; m < MROWS; ++m) acc[m] = warp_sum(acc[m]);
  // The next kernel's blocks may be scheduled now.  Not earlier: they would
  // share the SMs with this streaming pass while waiting for it to end.
  grid_launch_dependents();

  if (p.split_k == 1) {
    if (lane == 0 && j < p.N) {
#pragma unroll
      for (int m = 0; m < MROWS; ++m)
        if (m < p.M) write_out(p, out, prog, m, j, acc[m]);
    }
    return;
  }

  // Split-K: publish this split's partial sums, then the last CTA of the
  // row group reduces all splits in index order.
  float* partial = p.partial + z * p.split_k * p.M * static_cast<int64_t>(p.N);
  unsigned* counters = p.counters + z * gridDim.x;
  if (lane == 0 && j < p.N) {
#pragma unroll
    for (int m = 0; m < MROWS; ++m)
      if (m < p.M)
        partial[(static_cast<int64_t>(split) * p.M + m) * p.N + j] = acc[m];
  }
  __threadfence();
  __syncthreads();
  __shared__ unsigned s_is_last;
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&counters[blockIdx.x], 1u);
    s_is_last = (prev == static_cast<unsigned>(p.split_k - 1)) ? 1u : 0u;
  }
  __syncthreads();
  if (!s_is_last) return;
  __threadfence();
  // One thread per (m, row) of the group; splits added in order 0..split_k-1.
  for (int t = threadIdx.x; t < kGemvWarps * p.M; t += blockDim.x) {
    const int m = t / kGemvWarps;
    const int jj = blockIdx.x * kGemvWarps + (t % kGemvWarps);
    if (jj >= p.N) continue;
    const float s = sum_splits(partial + static_cast<int64_t>(m) * p.N + jj,
                               static_cast<int64_t>(p.M) * p.N, p.split_k);
    write_out(p, out, prog, m, jj, s);
  }
  if (threadIdx.x == 0) counters[blockIdx.x] = 0u;  // ready for the next launch
}

// Split-K inside a thread-block cluster (2 <= split <= 8): the CTAs of a row
// group's splits form one cluster along grid.y.  Each CTA streams its K
// range (eight 256-element steps in flight per lane, so that a split of up
// to 2048 K costs one memory round trip), then stores its warps' sums into
// the shared memory of the CTA of rank 0 (distributed shared memory) and
// leaves; rank 0 waits for every split's sums, adds them in split order,
// applies the epilogue and stores D.  No partial sums go to global memory,
// no arrival counter is needed, and of the cluster barrier's two phases the
// first (every CTA has started, so rank 0's shared memory may be written)
// completes while the splits stream; only rank 0 waits at the second.  The
// order of the additions is fixed, so results are bit-stable from run to
// run.  (Reading the other splits' sums from rank 0 after a full cluster
// barrier, with a second one keeping them resident, took 0.85 us more.)
constexpr int kGemvClusterUnroll = 8;
constexpr int kGemvClusterMax = 8;  // portable cluster size

template <int MROWS>
__global__ void __launch_bounds__(kGemvWarps * 32)
    gemv_cluster_kernel(const GemvParams p, const __grid_constant__ EpiProgram prog,
                        const GemvBatch bt) {
  __shared__ float part[kGemvClusterMax][MROWS][kGemvWarps];  // rank 0's: every split's sums
  cluster_arrive_relaxed();  // phase 1: this CTA has started
  grid_dependency_wait();  // launched as a dependent of the previous kernel
  const int64_t z = blockIdx.z;
  const __half* A = p.A + z * bt.sa;
  const __half* B = p.B + z * bt.sb;
  const GemvOut out{p.C + z * bt.sc, p.D + z * bt.sd, p.bias ? p.bias + z * bt.sbias : nullptr};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.x * kGemvWarps + warp;
  const int split = blockIdx.y;  // = the CTA's rank in its cluster
  const int k0 = split * p.k_chunk;
  const int k1 = min(p.K, k0 + p.k_chunk);

  float acc[MROWS];
  gemv_accumulate<MROWS, kGemvClusterUnroll>(p, A, B, j, lane, k0, k1, acc);
#pragma unroll
  for (int m = 0; m < MROWS; ++m) acc[m] = warp_sum(acc[m]);
  grid_launch_dependents();
  cluster_wait_acquire();  // every CTA of the cluster has started
  if (lane == 0) {
#pragma unroll
    for (int m = 0; m < MROWS; ++m)
      st_shared_cluster_f32(mapa_shared(smem_addr(&part[split][m][warp]), 0), acc[m]);
  }
  cluster_arrive_release();  // phase 2: this split's sums are in rank 0
  if (split != 0) return;
  cluster_wait_acquire();
  for (int t = threadIdx.x; t < kGemvWarps * p.M; t += blockDim.x) {
    const int m = t / kGemvWarps, w = t % kGemvWarps;
    const int jj = blockIdx.x * kGemvWarps + w;
    float sum = 0.0f;
#pragma unroll
    for (int r = 0; r < kGemvClusterMax; ++r)
      if (r < p.split_k) sum += part[r][m][w];
    if (jj < p.N) write_out(p, out, prog, m, jj, sum);
  }
}

// K == 0: D = epilogue(beta * C), no product term.  Element i of the M x N
// result is row i / N, column i % N.
__global__ void epilogue_only_kernel(int64_t M, int64_t N, const __half* C, int64_t ldc,
                                     __half* D, int64_t ldd, const __half* bias,
                                     const Epi epi, const __grid_constant__ EpiProgram prog) {
  grid_dependency_wait();  // launched as a dependent of the previous kernel
  const int64_t total = M * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t m = i / N, j = i - m * N;
    const float c = (epi.beta != 0.0f) ? __half2float(C[m * ldc + j]) : 0.0f;
    const float b = (epi.flags & kEpiBias) ? __half2float(bias[j]) : 0.0f;
    epi_store(D, m * ldd + j, epi_apply(0.0f, c, b, epi, prog), epi, prog);
  }
}

// K == 0 on the integer path: D = beta * C (mod 2^32).
__global__ void epilogue_only_i32_kernel(int64_t M, int64_t N, const int32_t* C, int64_t ldc,
                                         int32_t* D, int64_t ldd, int32_t beta) {
  grid_dependency_wait();  // launched as a dependent of the previous kernel
  const int64_t total = M * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t m = i / N, j = i - m * N;
    const uint32_t c = (beta != 0) ? static_cast<uint32_t>(C[m * ldc + j]) : 0u;
    D[m * ldd + j] = static_cast<int32_t>(static_cast<uint32_t>(beta) * c);
  }
}

// ------------------------------------------------------------ warp-MMA GEMV
// For 2 <= M <= 16 the FMA kernel above runs out of issue slots before HBM
// runs out of bandwidth (every B element meets M multiply-adds plus its
// conversion).  This variant feeds the same stream of B rows to warp-level
// m16n8k16 tensor-core MMAs: a warp owns 8 output columns (the MMA's n = 8)
// and up to 16 rows of A (its m = 16; rows >= M are zero), a CTA owns 64
// columns, and K is split over grid.y with the FMA kernel's deterministic
// last-CTA reduction.
//
// Fragments without shuffles: lane (g = lane / 4, t = lane % 4) loads 16
// bytes of B row n0 + g and of A rows g and g + 8 at k = k_step + 8t.  The
// m16n8k16 fragment wants, at lane (g, t), B[k][g] and A[g][k] for MMA-k
// 2t, 2t+1 (first register) and 2t+8, 2t+9 (second); taking MMA-k
// {2t, 2t+1, 2t+8, 2t+9} to mean k_step + 8t + {0, 1, 2, 3} in the first MMA
// and + {4, 5, 6, 7} in the second is one permutation of the 32 k of the step,
// the same for A and B, so the sum over k is unchanged.
constexpr int kMmaWarps = 8;
constexpr int kMmaCols = kMmaWarps * 8;  // output columns per CTA
constexpr int kMmaUnroll = 8;            // 32-wide k steps per batch

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Both MMAs of one 32-wide k step: A rows g (av) and g + 8 (av8), B row (bv).
__device__ __forceinline__ void mma_step(float (&d)[4], const uint4& av, const uint4& av8,
                                         const uint4& bv) {
  mma_16816(d, av.x, av8.x, av.y, av8.y, bv.x, bv.y);
  mma_16816(d, av.z, av8.z, av.w, av8.w, bv.z, bv.w);
}

// The 8 halves at row + k .. k + 7 that lie below k1, zeros above.
__device__ __forceinline__ uint4 load8_tail(const __half* row, int k, int k1) {
  uint4 v = make_uint4(0, 0, 0, 0);
  __half* h = reinterpret_cast<__half*>(&v);
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (k + e < k1) h[e] = row[k + e];
  return v;
}

template <int MROWS>  // 8: rows g only; 16: rows g and g + 8
__global__ void __launch_bounds__(kMmaWarps * 32)
    gemv_mma_kernel(const GemvParams p, const __grid_constant__ EpiProgram prog,
                    const GemvBatch bt) {
  grid_dependency_wait();  // launched as a dependent of the previous kernel
  const int64_t z = blockIdx.z;
  const GemvGroupProblem* gp = bt.group ? bt.group + z : nullptr;
  const int M = gp ? static_cast<int>(gp->M) : p.M;
  if (M == 0) return;  // an empty problem of a group (the whole block)
  const __half* A = gp ? gp->A : p.A + z * bt.sa;
  const __half* B = gp ? gp->B : p.B + z * bt.sb;
  const GemvOut out = gp ? GemvOut{gp->CD, gp->CD, gp->bias}
                         : GemvOut{p.C + z * bt.sc, p.D + z * bt.sd,
                                   p.bias ? p.bias + z * bt.sbias : nullptr};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int n0 = (blockIdx.x * kMmaWarps + warp) * 8;
  const int split = blockIdx.y;
  const int k0 = split * p.k_chunk;
  const int k1 = min(p.K, k0 + p.k_chunk);

  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  // Lanes past the last column read row N - 1 (in bounds) and discard it.
  const __half* brow = B + static_cast<int64_t>(min(n0 + g, p.N - 1)) * p.ldb;
  const bool has_a0 = g < M, has_a8 = MROWS == 16 && g + 8 < M;
  const __half* arow0 = A + static_cast<int64_t>(has_a0 ? g : 0) * p.lda;
  const __half* arow8 = A + static_cast<int64_t>(has_a8 ? g + 8 : 0) * p.lda;
  const uint4 zero = make_uint4(0, 0, 0, 0);

  if (n0 < p.N && k0 < k1) {  // warp-uniform: every lane reaches every MMA
    constexpr int kStep = 32;
    int kw = k0;  // the warp's k; this lane's 8 elements start at kw + 8t
    for (; kw + kMmaUnroll * kStep <= k1; kw += kMmaUnroll * kStep) {
      uint4 bv[kMmaUnroll], av[kMmaUnroll], av8[kMmaUnroll];
#pragma unroll
      for (int u = 0; u < kMmaUnroll; ++u) bv[u] = ld_stream(brow + kw + u * kStep + 8 * t);
#pragma unroll
      for (int u = 0; u < kMmaUnroll; ++u) {
        av[u] = has_a0 ? __ldg(reinterpret_cast<const uint4*>(arow0 + kw + u * kStep + 8 * t))
                       : zero;
        av8[u] = has_a8 ? __ldg(reinterpret_cast<const uint4*>(arow8 + kw + u * kStep + 8 * t))
                        : zero;
      }
#pragma unroll
      for (int u = 0; u < kMmaUnroll; ++u) mma_step(acc, av[u], av8[u], bv[u]);
    }
    // whole 32-wide steps left
    for (; kw + kStep <= k1; kw += kStep) {
      const uint4 bv = ld_stream(brow + kw + 8 * t);
      const uint4 av =
          has_a0 ? __ldg(reinterpret_cast<const uint4*>(arow0 + kw + 8 * t)) : zero;
      const uint4 av8 =
          has_a8 ? __ldg(reinterpret_cast<const uint4*>(arow8 + kw + 8 * t)) : zero;
      mma_step(acc, av, av8, bv);
    }
    // a last partial step: elements at or past k1 read as zero
    if (kw < k1) {
      const int kl = kw + 8 * t;
      const uint4 bv = load8_tail(brow, kl, k1);
      const uint4 av = has_a0 ? load8_tail(arow0, kl, k1) : zero;
      const uint4 av8 = has_a8 ? load8_tail(arow8, kl, k1) : zero;
      mma_step(acc, av, av8, bv);
    }
  }
  // The next kernel's blocks may be scheduled now (see the FMA kernel).
  grid_launch_dependents();

  // acc[0..1]: row g, columns n0 + 2t + {0, 1}; acc[2..3]: row g + 8.
  const int col = n0 + 2 * t;
  if (p.split_k == 1) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        if (g + 8 * h < M && col + e < p.N)
          write_out(p, out, prog, g + 8 * h, col + e, acc[2 * h + e]);
    return;
  }

  // Split-K: partials, then the last CTA of the column group reduces.
  // problem z's partials: [split][M][N] inside a slot of split x p.M x N
  float* partial = p.partial + z * p.split_k * p.M * static_cast<int64_t>(p.N);
  unsigned* counters = p.counters + z * gridDim.x;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int e = 0; e < 2; ++e)
      if (g + 8 * h < M && col + e < p.N)
        partial[(static_cast<int64_t>(split) * M + g + 8 * h) * p.N + col + e] = acc[2 * h + e];
  __threadfence();
  __syncthreads();
  __shared__ unsigned s_is_last;
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&counters[blockIdx.x], 1u);
    s_is_last = (prev == static_cast<unsigned>(p.split_k - 1)) ? 1u : 0u;
  }
  __syncthreads();
  if (!s_is_last) return;
  __threadfence();
  for (int i = threadIdx.x; i < kMmaCols * M; i += blockDim.x) {
    const int m = i / kMmaCols;
    const int jj = blockIdx.x * kMmaCols + (i % kMmaCols);
    if (jj >= p.N) continue;
    const float s = sum_splits(partial + static_cast<int64_t>(m) * p.N + jj,
                               static_cast<int64_t>(M) * p.N, p.split_k);
    write_out(p, out, prog, m, jj, s);
  }
  if (threadIdx.x == 0) counters[blockIdx.x] = 0u;  // ready for the next launch
}

// One CTA waits on a barrier nobody arrives on; the bounded wait must give up,
// record the timeout and let the kernel exit normally.
__global__ void wait_selftest_kernel(int* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_wait(&bar, 0, timeout_ns, status);
  }
  __syncthreads();
}

}  // namespace

// Splits of 2 .. 8 reduce inside a cluster and need no workspace.
bool gemv_split_in_cluster(int split) { return split >= 2 && split <= kGemvClusterMax; }

int64_t gemv_partial_elems(const dg_tile_plan& plan, int64_t M, int64_t N, int64_t batch) {
  if (plan.kernel == DG_KERNEL_GEMV && gemv_split_in_cluster(plan.split_k)) return 0;
  return plan.split_k > 1 ? static_cast<int64_t>(plan.split_k) * M * N * batch : 0;
}

int64_t gemv_counter_elems(const dg_tile_plan& plan, int64_t N, int64_t batch) {
  if (plan.kernel == DG_KERNEL_GEMV && gemv_split_in_cluster(plan.split_k)) return 0;
  return plan.split_k > 1 ? (N + kGemvWarps - 1) / kGemvWarps * batch : 0;
}

int gemv_kernel_regs(int64_t M, int split) {
  static std::atomic<int> slot[8] = {{-1}, {-1}, {-1}, {-1}, {-1}, {-1}, {-1}, {-1}};
  if (gemv_split_in_cluster(split)) {
    if (M <= 1) return kernel_regs(gemv_cluster_kernel<1>, slot[4]);
    if (M <= 2) return kernel_regs(gemv_cluster_kernel<2>, slot[5]);
    if (M <= 4) return kernel_regs(gemv_cluster_kernel<4>, slot[6]);
    return kernel_regs(gemv_cluster_kernel<kGemvMaxM>, slot[7]);
  }
  if (M <= 1) return kernel_regs(gemv_splitk_kernel<1>, slot[0]);
  if (M <= 2) return kernel_regs(gemv_splitk_kernel<2>, slot[1]);
  if (M <= 4) return kernel_regs(gemv_splitk_kernel<4>, slot[2]);
  return kernel_regs(gemv_splitk_kernel<kGemvMaxM>, slot[3]);
}

int gemv_mma_kernel_regs(int64_t M) {
  static std::atomic<int> slot[2] = {{-1}, {-1}};
  return M <= 8 ? kernel_regs(gemv_mma_kernel<8>, slot[0])
                : kernel_regs(gemv_mma_kernel<16>, slot[1]);
}

cudaError_t launch_gemv(const GemmArgs& a, const dg_tile_plan& plan, const SplitKWorkspace& ws) {
  GemvParams p;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.A = static_cast<const __half*>(a.A);
  p.lda = a.lda;
  p.B = static_cast<const __half*>(a.B);
  p.ldb = a.ldb;
  p.C = static_cast<const __half*>(a.C);
  p.ldc = a.ldc;
  p.D = static_cast<__half*>(a.D);
  p.ldd = a.ldd;
  p.bias = static_cast<const __half*>(a.bias);
  p.epi = make_epi(a);
  p.split_k = plan.split_k;
  p.k_chunk = plan.k_tile;
  p.partial = ws.partial;
  p.counters = ws.counters;
  const dim3 grid(static_cast<unsigned>((a.N + kGemvWarps - 1) / kGemvWarps),
                  static_cast<unsigned>(plan.split_k));
  const dim3 block(kGemvWarps * 32);
  const bool cluster = gemv_split_in_cluster(plan.split_k);
  auto kern = cluster ? (a.M <= 1   ? gemv_cluster_kernel<1>
                         : a.M <= 2 ? gemv_cluster_kernel<2>
                         : a.M <= 4 ? gemv_cluster_kernel<4>
                                    : gemv_cluster_kernel<kGemvMaxM>)
                      : (a.M <= 1   ? gemv_splitk_kernel<1>
                         : a.M <= 2 ? gemv_splitk_kernel<2>
                         : a.M <= 4 ? gemv_splitk_kernel<4>
                                    : gemv_splitk_kernel<kGemvMaxM>);
  // grid.z takes at most 65535 problems per launch
  constexpr int64_t kMaxZ = 65535;
  const int64_t groups = (a.N + kGemvWarps - 1) / kGemvWarps;
  const GemvBatch bt{a.stride_a, a.stride_b, a.stride_c, a.stride_d, a.stride_bias};
  for (int64_t z0 = 0; z0 < a.batch; z0 += kMaxZ) {
    const int64_t nz = std::min(kMaxZ, a.batch - z0);
    GemvParams q = p;
    q.A += z0 * bt.sa;
    q.B += z0 * bt.sb;
    q.C += z0 * bt.sc;
    q.D += z0 * bt.sd;
    if (q.bias) q.bias += z0 * bt.sbias;
    if (q.partial) q.partial += z0 * plan.split_k * a.M * a.N;
    if (q.counters) q.counters += z0 * groups;
    const dim3 g(grid.x, grid.y, static_cast<unsigned>(nz));
    cudaError_t e;
    if (cluster) {
      // the splits of a row group as one cluster along y
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = g;
      cfg.blockDim = block;
      cfg.stream = a.stream;
      cudaLaunchAttribute attr[2];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 1;
      attr[0].val.clusterDim.y = static_cast<unsigned>(plan.split_k);
      attr[0].val.clusterDim.z = 1;
      attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[1].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 2;
      e = cudaLaunchKernelEx(&cfg, kern, q, make_program(a), bt);
    } else {
      e = launch_dependent(kern, g, block, 0, a.stream, q, make_program(a), bt);
    }
    count_launches(1);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_gemv_mma(const GemmArgs& a, const dg_tile_plan& plan,
                            const SplitKWorkspace& ws) {
  if (a.M < 1 || a.M > 16) return cudaErrorInvalidValue;
  GemvParams p;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.A = static_cast<const __half*>(a.A);
  p.lda = a.lda;
  p.B = static_cast<const __half*>(a.B);
  p.ldb = a.ldb;
  p.C = static_cast<const __half*>(a.C);
  p.ldc = a.ldc;
  p.D = static_cast<__half*>(a.D);
  p.ldd = a.ldd;
  p.bias = static_cast<const __half*>(a.bias);
  p.epi = make_epi(a);
  p.split_k = plan.split_k;
  p.k_chunk = plan.k_tile;
  p.partial = ws.partial;
  p.counters = ws.counters;
  const unsigned gx = static_cast<unsigned>((a.N + kMmaCols - 1) / kMmaCols);
  auto kern = a.M <= 8 ? gemv_mma_kernel<8> : gemv_mma_kernel<16>;
  constexpr int64_t kMaxZ = 65535;
  const GemvBatch bt{a.stride_a, a.stride_b, a.stride_c, a.stride_d, a.stride_bias};
  for (int64_t z0 = 0; z0 < a.batch; z0 += kMaxZ) {
    const int64_t nz = std::min(kMaxZ, a.batch - z0);
    GemvParams q = p;
    q.A += z0 * bt.sa;
    q.B += z0 * bt.sb;
    q.C += z0 * bt.sc;
    q.D += z0 * bt.sd;
    if (q.bias) q.bias += z0 * bt.sbias;
    if (q.partial) q.partial += z0 * plan.split_k * a.M * a.N;
    if (q.counters) q.counters += z0 * gx;
    const dim3 grid(gx, static_cast<unsigned>(plan.split_k), static_cast<unsigned>(nz));
    const cudaError_t e = launch_dependent(kern, grid, dim3(kMmaWarps * 32), 0, a.stream, q,
                                           make_program(a), bt);
    count_launches(1);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_gemv_mma_grouped(const GemmArgs& a, const void* table, int64_t count,
                                    int64_t max_m, const dg_tile_plan& plan,
                                    const SplitKWorkspace& ws) {
  if (max_m < 1 || max_m > 16 || count < 1) return cudaErrorInvalidValue;
  GemvParams p{};
  p.M = static_cast<int>(max_m);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.lda = a.lda;
  p.ldb = a.ldb;
  p.ldc = a.N;
  p.ldd = a.N;
  p.epi = make_epi(a);
  p.split_k = plan.split_k;
  p.k_chunk = plan.k_tile;
  p.partial = ws.partial;
  p.counters = ws.counters;
  const unsigned gx = static_cast<unsigned>((a.N + kMmaCols - 1) / kMmaCols);
  auto kern = max_m <= 8 ? gemv_mma_kernel<8> : gemv_mma_kernel<16>;
  constexpr int64_t kMaxZ = 65535;
  const auto* group = static_cast<const GemvGroupProblem*>(table);
  for (int64_t z0 = 0; z0 < count; z0 += kMaxZ) {
    const int64_t nz = std::min(kMaxZ, count - z0);
    GemvParams q = p;
    if (q.partial) q.partial += z0 * plan.split_k * max_m * a.N;
    if (q.counters) q.counters += z0 * gx;
    const GemvBatch bt{0, 0, 0, 0, 0, group + z0};
    const dim3 grid(gx, static_cast<unsigned>(plan.split_k), static_cast<unsigned>(nz));
    const cudaError_t e = launch_dependent(kern, grid, dim3(kMmaWarps * 32), 0, a.stream, q,
                                           make_program(a), bt);
    count_launches(1);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int64_t gemv_group_entry_bytes() { return sizeof(GemvGroupProblem); }

void gemv_group_entry(void* table, int64_t i, const void* A, const void* B, void* CD,
                      const void* bias, int64_t M) {
  static_cast<GemvGroupProblem*>(table)[i] =
      GemvGroupProblem{static_cast<const __half*>(A), static_cast<const __half*>(B),
                       static_cast<__half*>(CD), static_cast<const __half*>(bias), M};
}

cudaError_t launch_epilogue_only(const GemmArgs& a) {
  const int64_t total = a.M * a.N;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(a.sm_count) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaError_t e;
  if (a.dtype_a == DG_I8) {
    e = launch_dependent(epilogue_only_i32_kernel, dim3(static_cast<unsigned>(blocks)),
                         dim3(threads), 0, a.stream, a.M, a.N, static_cast<const int32_t*>(a.C),
                         a.ldc, static_cast<int32_t*>(a.D), a.ldd, static_cast<int32_t>(a.beta));
  } else {
    e = launch_dependent(epilogue_only_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads),
                         0, a.stream, a.M, a.N, static_cast<const __half*>(a.C), a.ldc,
                         static_cast<__half*>(a.D), a.ldd, static_cast<const __half*>(a.bias),
                         make_epi(a), make_program(a));
  }
  count_launches(1);
  return e;
}

cudaError_t launch_wait_selftest(cudaStream_t stream, int* status, uint64_t timeout_ns) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  count_launches(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Split-K scratch for callers that cannot allocate device memory.
//
// dg_gemm grows a cudaMalloc'd workspace the first time a shape needs split-K
// partials.  Some callers cannot let a library call cudaMalloc: code running
// while a CUDA graph is being captured, inference runtimes that hand out every
// byte of device memory from their own pool, or hosts whose allocator is
// locked down.  dg_gemm_thin_noalloc runs the same GEMV kernel with its
// partial sums and arrival counters in this fixed, file-scope device array
// instead.  Every GPU that loads the library holds these bytes until the
// process exits.
constexpr size_t kNoAllocCounterBytes = 64 * 1024;        // 16384 row-group counters
constexpr size_t kNoAllocPartialBytes = 2 * 1024 * 1024;  // 524288 FP32 partial sums
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocCounterBytes +
                                                                 kNoAllocPartialBytes];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};
dg_hw_desc g_noalloc_hw[kNoAllocMaxDevices] = {};

// Device address of the scratch array on `dev` (which must be current) and
// that device's description.  The host-side name of the array is only a
// stand-in, so the address is looked up once per device with
// cudaGetSymbolAddress; the description (a dozen attribute queries) is
// filled at the same time, so later calls make no query at all.
dg_status noalloc_setup(int dev, void** out, dg_hw_desc* hw) {
  if (dev < 0 || dev >= kNoAllocMaxDevices)
    return set_error(DG_ERR_INVALID_STATE, "device index beyond the scratch table");
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    dg_hw_desc h{};
    const dg_status s = fill_hw_desc(dev, &h);
    if (s != DG_OK) return s;
    if (h.cc_major != 10 || h.cc_minor != 3)
      return set_error(DG_ERR_INVALID_STATE, "libdg is built for sm_103a (GB300) only");
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return set_error(DG_ERR_CUDA, "cudaGetSymbolAddress of the static split-K scratch failed");
    }
    g_noalloc_hw[dev] = h;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  *hw = g_noalloc_hw[dev];
  return DG_OK;
}
}  // namespace

}  // namespace dg

using namespace dg;

extern "C" dg_status dg_gemm_thin_noalloc(int64_t M, int64_t N, int64_t K, dg_dtype dtype_a,
                                          dg_dtype dtype_b, const void* A, int64_t lda,
                                          const void* B, int64_t ldb, void* C, const void* bias,
                                          float alpha, float beta, dg_epilogue epilogue,
                                          dg_stream_t stream) {
  clear_error();
  dg_status s = validate_gemm_args(M, N, K, dtype_a, dtype_b, A, lda, B, ldb, C, bias, alpha,
                                   beta, epilogue);
  if (s != DG_OK) return s;
  if (M == 0 || N == 0) return DG_OK;
  if (dtype_a != DG_F16 || dtype_b != DG_F16 || M > kGemvMaxM)
    return set_error(DG_ERR_UNSUPPORTED, "dg_gemm_thin_noalloc takes F16 x F16 with M <= 8");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return set_error(DG_ERR_INVALID_STATE, "no current CUDA device");
  }
  dg_hw_desc hw{};
  void* scratch = nullptr;
  s = noalloc_setup(dev, &scratch, &hw);
  if (s != DG_OK) return s;

  // The split-K GEMV's own best split (the fastest GEMV candidate of the
  // planner; dg_gemm may pick another kernel or split for the same shape).
  int64_t chunk = 0;
  const int split = gemv_best_split(M, N, K, hw, &chunk);
  const int64_t row_groups = (N + kGemvWarps - 1) / kGemvWarps;
  const int64_t partial_bytes = split > 1 ? static_cast<int64_t>(split) * M * N * 4 : 0;
  const int64_t counter_bytes = split > 1 ? row_groups * 4 : 0;
  if (partial_bytes > static_cast<int64_t>(kNoAllocPartialBytes) ||
      counter_bytes > static_cast<int64_t>(kNoAllocCounterBytes)) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "shape needs %lld bytes of split-K partials and %lld bytes of counters; the static "
             "scratch holds %zu and %zu",
             (long long)partial_bytes, (long long)counter_bytes, kNoAllocPartialBytes,
             kNoAllocCounterBytes);
    return set_error(DG_ERR_INVALID_ARG, msg);
  }

  unsigned* counters = static_cast<unsigned*>(scratch);
  float* partial =
      reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + kNoAllocCounterBytes);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (split > 1) {
    // The array keeps the previous call's contents; counters must start at zero.
    e = cudaMemsetAsync(counters, 0, static_cast<size_t>(counter_bytes), st);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return set_error(DG_ERR_CUDA, "cudaMemsetAsync of the scratch counters failed");
    }
  }

  GemmArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.dtype_a = dtype_a;
  a.dtype_b = dtype_b;
  a.A = A;
  a.lda = lda;
  a.B = B;
  a.ldb = ldb;
  a.C = C;
  a.ldc = N;
  a.D = C;
  a.ldd = N;
  a.bias = bias;
  a.alpha = alpha;
  a.beta = beta;
  a.epi = ((epilogue == DG_EPI_BIAS || epilogue == DG_EPI_BIAS_GELU) ? kEpiBias : 0) |
          ((epilogue == DG_EPI_GELU || epilogue == DG_EPI_BIAS_GELU) ? kEpiGelu : 0);
  a.n_ops = 0;
  a.batch = 1;
  a.stride_a = a.stride_b = a.stride_c = a.stride_d = a.stride_bias = 0;
  a.stream = st;
  a.status = nullptr;
  a.timeout_ns = 0;
  a.exact_i32 = false;
  a.sm_count = hw.sm_count;
  dg_tile_plan plan{};
  plan.kernel = DG_KERNEL_GEMV;
  plan.split_k = split;
  plan.k_tile = static_cast<int>(chunk);
  SplitKWorkspace ws{partial, partial_bytes / 4, counters, counter_bytes / 4};
  e = launch_gemv(a, plan, ws);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return set_error(DG_ERR_CUDA, "GEMV launch failed");
  }
  return DG_OK;
}
