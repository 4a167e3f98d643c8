// Dense FP16 GEMM on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
//   D[M x N] = epilogue(alpha * A[M x K] . B[N x K]^T + beta * C)
//
// The contraction the "DeepGEMM" articles build their tile planner around
// (discosf.com/news/5532976, section 3.2: a 4096^3 FP16 GEMM; section 3.5:
// FP32 accumulation, FP16 output; kwkr.cn/news/562171, section 2.2 first and
// third layers: planned tiles and a fused epilogue).  The pages target
// warp-level mma.sync on A100/H100; on Blackwell the same contraction maps to
// a single-thread-issued tcgen05.mma with the accumulator in tensor memory:
//
//   warp 0      TMA producer: a ring of `Stages` shared-memory slots, each a
//               128 x 64 tile of A and a BN x 64 tile of B (128-byte swizzle);
//   warp 1      MMA issuer: 4 x tcgen05.mma (K = 16 each) per slot into a
//               128 x BN FP32 accumulator in TMEM; tcgen05.commit frees slots;
//   warp 2      allocates / frees the tensor memory (2 accumulators);
//   warps 4-7   epilogue: tcgen05.ld of the accumulator (each warp owns 32 of
//               the 128 TMEM lanes = rows), alpha/beta/bias/GELU in FP32,
//               FP16 round-to-nearest-even, stored straight to D.
//
// The kernel is persistent (one CTA per SM walks the tile list), and the two
// TMEM accumulators let the epilogue of tile i overlap the main loop of tile
// i+1.  Out-of-range rows and K columns are zero-filled by TMA; the epilogue
// masks rows >= M and columns >= N.  Every mbarrier wait is bounded: on a
// timeout the CTA records it in the status word, drains its own copies and
// MMAs, frees its tensor memory and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tc_common.cuh"

namespace dg {
namespace {

using tc::kBlockK;
using tc::kBlockM;
constexpr int kThreads = 256;
constexpr int kEpiWarp0 = 4;
constexpr int kTileBytesA = kBlockM * kBlockK * 2;

struct TcParams {
  int M, N, K;
  int num_m_blocks, num_n_blocks, num_tiles, num_k_blocks;
  int group_m;
  Epi epi;
  __half* CD;  // C in / D out, leading dimension N
  const __half* bias;
  int* status;
  uint64_t timeout_ns;
};

template <int BN, int Stages>
struct TcSmem {
  static constexpr int kTileBytesB = BN * kBlockK * 2;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + Stages * kTileBytesA;
  static constexpr int kOffBar = kOffB + Stages * kTileBytesB;
  // full[Stages], empty[Stages], tmem_full[2], tmem_empty[2], drain
  static constexpr int kNumBars = 2 * Stages + 5;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kBytes = kOffAbort + 4;
  static constexpr int kLaunchBytes = kBytes + 1024;  // room to align the base to 1 KB
};

__device__ __forceinline__ bool aborted(volatile int* flag) { return *flag != 0; }

template <int BN, int Stages>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_f16_tc_kernel(const __grid_constant__ CUtensorMap tmap_a,
                       const __grid_constant__ CUtensorMap tmap_b, const TcParams p) {
  using L = TcSmem<BN, Stages>;
  constexpr int kTmemCols = 2 * BN;
  constexpr uint32_t kIdesc = idesc_f16_f32(kBlockM, BN);
  constexpr uint32_t kStageTx = kTileBytesA + L::kTileBytesB;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* smem_a = smem + L::kOffA;
  uint8_t* smem_b = smem + L::kOffB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + Stages;
  uint64_t* tmem_full = bars + 2 * Stages;
  uint64_t* tmem_empty = bars + 2 * Stages + 2;
  uint64_t* drain_bar = bars + 2 * Stages + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], 4 * 32);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 2) tmem_alloc<kTmemCols>(tmem_slot);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one_lane()) {
      const uint64_t pol = policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        int m_blk, n_blk;
        tc::tile_coords(t, p.num_m_blocks, p.num_n_blocks, p.group_m, m_blk, n_blk);
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          if (aborted(abort_flag) ||
              !mbar_wait(&empty_bar[stage], phase ^ 1, p.timeout_ns, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[stage], kStageTx);
          tma_load_2d(&tmap_a, &full_bar[stage], smem_a + stage * kTileBytesA, kb * kBlockK,
                      m_blk * kBlockM, pol);
          tma_load_2d(&tmap_b, &full_bar[stage], smem_b + stage * L::kTileBytesB, kb * kBlockK,
                      n_blk * BN, pol);
          ++issued;
          if (++stage == Stages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        // Let the copies this thread started land before the CTA goes away.
        const int64_t first = issued > Stages ? issued - Stages : 0;
        for (int64_t i = first; i < issued; ++i)
          mbar_wait(&full_bar[i % Stages], static_cast<uint32_t>((i / Stages) & 1), p.timeout_ns,
                    p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one_lane()) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        if (aborted(abort_flag) ||
            !mbar_wait(&tmem_empty[acc], acc_phase ^ 1, p.timeout_ns, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          if (aborted(abort_flag) ||
              !mbar_wait(&full_bar[stage], phase, p.timeout_ns, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a0 = smem_addr(smem_a + stage * kTileBytesA);
          const uint32_t b0 = smem_addr(smem_b + stage * L::kTileBytesB);
#pragma unroll
          for (int k = 0; k < kBlockK / 16; ++k) {
            tc_mma_f16(d_tmem, smem_desc_sw128(a0 + k * 32), smem_desc_sw128(b0 + k * 32), kIdesc,
                       (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit(&empty_bar[stage]);
          if (++stage == Stages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&tmem_full[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        // Wait for the MMAs already issued before the tensor memory is freed.
        tc_commit(drain_bar);
        mbar_wait(drain_bar, 0, p.timeout_ns, p.status);
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - kEpiWarp0;  // TMEM lanes 32*ew .. 32*ew+31
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int m_blk, n_blk;
      tc::tile_coords(t, p.num_m_blocks, p.num_n_blocks, p.group_m, m_blk, n_blk);
      if (aborted(abort_flag) ||
          !mbar_wait(&tmem_full[acc], acc_phase, p.timeout_ns, p.status)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after_sync();
      const int row = m_blk * kBlockM + ew * 32 + lane;
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32cols(tbase + c * 32, r);
        tc_wait_ld();
        const int col0 = n_blk * BN + c * 32;
        if (col0 < p.N) tc::epilogue_f16_chunk(r, row, col0, p.M, p.N, p.epi, p.CD, p.bias);
      }
      tc_fence_before_sync();
      mbar_arrive(&tmem_empty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after_sync();
    tmem_dealloc<kTmemCols>(tmem_base);
  }
}

template <int BN, int Stages>
cudaError_t run_tc(const GemmArgs& a, const dg_tile_plan& plan) {
  using L = TcSmem<BN, Stages>;
  CUtensorMap ta, tb;
  cudaError_t e = tc::make_f16_kmajor_map(&ta, a.A, a.M, a.K, a.lda, kBlockM);
  if (e != cudaSuccess) return e;
  e = tc::make_f16_kmajor_map(&tb, a.B, a.N, a.K, a.ldb, BN);
  if (e != cudaSuccess) return e;

  TcParams p;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.num_m_blocks = static_cast<int>((a.M + kBlockM - 1) / kBlockM);
  p.num_n_blocks = static_cast<int>((a.N + BN - 1) / BN);
  p.num_tiles = p.num_m_blocks * p.num_n_blocks;
  p.num_k_blocks = static_cast<int>((a.K + kBlockK - 1) / kBlockK);
  p.group_m = 16;
  p.epi = Epi{a.alpha, a.beta, a.epi};
  p.CD = static_cast<__half*>(a.C);
  p.bias = static_cast<const __half*>(a.bias);
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;

  auto kern = gemm_f16_tc_kernel<BN, Stages>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kLaunchBytes);
  if (e != cudaSuccess) return e;
  int grid = plan.grid > 0 ? plan.grid : a.sm_count;
  if (grid > p.num_tiles) grid = p.num_tiles;
  kern<<<grid, kThreads, L::kLaunchBytes, a.stream>>>(ta, tb, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

// Tile shapes compiled into the library; the planner only proposes these.
cudaError_t launch_tc(const GemmArgs& a, const dg_tile_plan& plan) {
  if (a.dtype_a != DG_F16 || a.dtype_b != DG_F16) return cudaErrorNotSupported;
  switch (plan.n_tile) {
    case 256:
      if (plan.stages == 4) return run_tc<256, 4>(a, plan);
      break;
    case 128:
      if (plan.stages == 6) return run_tc<128, 6>(a, plan);
      break;
    case 64:
      if (plan.stages == 8) return run_tc<64, 8>(a, plan);
      break;
  }
  return cudaErrorNotSupported;
}

}  // namespace dg
