// W4A16 GEMM with the packed 4-bit weights widened in tensor memory:
//
//   D[M x N] = epilogue(alpha * A[M x K] . B[N x K]^T + beta * C)
//
// A: FP16 activations; B: E2M1 weights packed two codes a byte (the
// {weight: int4_e2m1, activation: fp16, output: fp16} triple of
// discosf.com/news/5532976, section 2.2 layer 2, unpacked inside the kernel
// as section 4.3 asks); bias + GELU fused (kwkr.cn/news/562171, section 2.2
// third layer).
//
// There is no tensor-core kind that multiplies FP16 by 4-bit codes, and
// widened weights handed to the tensor core through shared memory cost a
// proxy fence per stage, about as long as the stage's MMAs.  The MMA's A
// operand may instead sit in tensor memory, which tcgen05.st fills and a
// tcgen05 fence hands over.  So the kernel computes D^T: the weights are the
// MMA's A (128 rows of B a tile, widened into tensor memory), the activations
// its B (TMA into shared memory, 128-byte swizzle), and the accumulator holds
// D^T with one weight row per tensor-memory lane:
//
//   warp 0          TMA producer: per stage the 32 bytes of codes of each of
//                   the tile's 128 weight rows (64 values of K) and the
//                   activation tile (BN rows x 64 values of K);
//   warps 12, 13,   converters, one per tensor-memory lane quarter (a warp
//   2, 3            reaches the lanes of its index mod 4): lane r of quarter
//                   q reads weight row 32 q + r's 32 bytes, widens them with
//                   cvt.rn.f16x2.e2m1x2 (exact; column j of the row holds K
//                   values 2j and 2j + 1, low nibble in the low half) and
//                   stores the 32 columns into an A slot with tcgen05.st;
//   warp 1          MMA issuer: tcgen05.mma kind::f16 with A in tensor
//                   memory, four of K = 16 per stage; commits free the stage's
//                   shared memory and the A slot;
//   warps 4-11      epilogue: lane = weight row n (a column of D), 32
//                   accumulator columns = 32 rows of D; each lane writes its
//                   column of a 32 x 32 box of D in shared memory and TMA
//                   stores the box;  warp 2 also allocates tensor memory.
//
// Tensor memory: two accumulators of BN columns, then (512 - 2 BN) / 32
// A slots of 32 columns (128 rows x 64 FP16 values).  The kernel is
// persistent (one CTA per SM walks the tiles).  Every mbarrier wait is
// bounded: on a timeout the CTA records it in the status word, drains its
// own copies and MMAs, frees its tensor memory and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "convert.cuh"
#include "tc_common.cuh"

namespace dg {
namespace {

using tc::kBlockK;  // 64 values of K per stage
using tc::kBlockM;  // 128 weight rows per tile (tensor-memory lanes)

constexpr int kThreads = 448;  // 14 warps
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 8;
constexpr int kBoxBytes = 32 * 32 * 2;  // a 32 x 32 FP16 box of D or C, rows of 64 bytes

// The lane quarter a converter warp widens, -1 for other warps.
__device__ __forceinline__ int converter_quarter(int warp) {
  return warp >= 12 ? warp - 12 : (warp == 2 || warp == 3 ? warp : -1);
}

struct W4tParams {
  int M, N, K;
  int num_w_blocks;  // tiles along N (128 weight rows each)
  int num_x_blocks;  // tiles along M (BN activation rows each)
  int num_tiles, num_k_blocks;
  Epi epi;
  const __half* bias;
  int* status;
  uint64_t timeout_ns;
};

template <int BN, int Stages>
struct W4tSmem {
  static constexpr int kASlots = (512 - 2 * BN) / 32;
  static constexpr int kXBytes = BN * kBlockK * 2;       // activation tile, swizzled rows
  static constexpr int kWBytes = kBlockM * kBlockK / 2;  // 32 bytes of codes per weight row
  static constexpr int kOffX = 0;
  static constexpr int kOffW = kOffX + Stages * kXBytes;
  static constexpr int kOffEpi = kOffW + Stages * kWBytes;
  static constexpr int kOffBar = kOffEpi + kEpiWarps * 2 * kBoxBytes;
  // x_full, w_full, empty [Stages]; a_full, a_empty [kASlots]; tmem_full,
  // tmem_empty [2]; drain; one C-load barrier per epilogue box
  static constexpr int kNumBars = 3 * Stages + 2 * kASlots + 5 + 2 * kEpiWarps;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kBytes = kOffAbort + 4;
  static constexpr int kLaunchBytes = kBytes + 1024;
  static_assert(kXBytes % 1024 == 0, "activation tiles keep the 1 KB swizzle alignment");
  static_assert(kASlots >= 2, "tensor memory for at least two A slots");
  static_assert(kBytes + 1024 <= 232448, "shared memory of one CTA");
};

__device__ __forceinline__ bool aborted(volatile int* flag) { return *flag != 0; }

// Tile t: the x (activation) block runs fastest.
__device__ __forceinline__ void w4t_coords(const W4tParams& p, int t, int& w_blk, int& x_blk) {
  w_blk = t / p.num_x_blocks;
  x_blk = t - w_blk * p.num_x_blocks;
}

template <int BN, int Stages>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_w4t_kernel(const __grid_constant__ CUtensorMap tmap_x,
                    const __grid_constant__ CUtensorMap tmap_w,
                    const __grid_constant__ CUtensorMap tmap_c,
                    const __grid_constant__ CUtensorMap tmap_d, const W4tParams p,
                    const __grid_constant__ EpiProgram prog) {
  using L = W4tSmem<BN, Stages>;
  constexpr int kSlots = L::kASlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* smem_x = smem + L::kOffX;
  uint8_t* smem_w = smem + L::kOffW;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* x_full = bars;
  uint64_t* w_full = bars + Stages;
  uint64_t* empty_bar = bars + 2 * Stages;
  uint64_t* a_full = bars + 3 * Stages;
  uint64_t* a_empty = a_full + kSlots;
  uint64_t* tmem_full = a_empty + kSlots;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* drain_bar = tmem_empty + 2;
  uint64_t* epi_bar = drain_bar + 1;  // [kEpiWarps][2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Stages; ++s) {
      mbar_init(&x_full[s], 1);
      mbar_init(&w_full[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&a_full[s], 4);  // the four converter warps
      mbar_init(&a_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], kEpiWarps * 32);
    }
    mbar_init(drain_bar, 1);
    for (int b = 0; b < 2 * kEpiWarps; ++b) mbar_init(&epi_bar[b], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_w);
    tma_prefetch_desc(&tmap_d);
    if (p.epi.beta != 0.0f) tma_prefetch_desc(&tmap_c);
  }
  if (warp == 2) tmem_alloc<512>(tmem_slot);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  bool ok = true;
  grid_dependency_wait();

  const int quarter = converter_quarter(warp);
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one_lane()) {
      const uint64_t pol = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        int w_blk, x_blk;
        w4t_coords(p, t, w_blk, x_blk);
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          if (!mbar_wait_abortable(&empty_bar[stage], phase ^ 1, p.timeout_ns, p.status,
                                   abort_flag)) {
            ok = false;
            break;
          }
          // codes first: the converters start on them while the activations land
          mbar_arrive_expect_tx(&w_full[stage], L::kWBytes);
          tma_load_2d(&tmap_w, &w_full[stage], smem_w + stage * L::kWBytes, kb * (kBlockK / 2),
                      w_blk * kBlockM, pol);
          mbar_arrive_expect_tx(&x_full[stage], L::kXBytes);
          tma_load_2d(&tmap_x, &x_full[stage], smem_x + stage * L::kXBytes, kb * kBlockK,
                      x_blk * BN, pol);
          ++issued;
          if (++stage == Stages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      grid_launch_dependents();
      if (!ok) {
        *abort_flag = 1;
        const int64_t first = issued > Stages ? issued - Stages : 0;
        for (int64_t i = first; i < issued; ++i) {
          const uint32_t par = static_cast<uint32_t>((i / Stages) & 1);
          mbar_wait(&w_full[i % Stages], par, p.timeout_ns, p.status);
          mbar_wait(&x_full[i % Stages], par, p.timeout_ns, p.status);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one_lane()) {
      const uint32_t idesc = idesc_f16_f32(kBlockM, BN);
      int stage = 0, slot = 0, acc = 0;
      uint32_t phase = 0, a_phase = 0, acc_phase = 0;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        if (!mbar_wait_abortable(&tmem_empty[acc], acc_phase ^ 1, p.timeout_ns, p.status,
                                 abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          if (!mbar_wait_abortable(&x_full[stage], phase, p.timeout_ns, p.status, abort_flag) ||
              !mbar_wait_abortable(&a_full[slot], a_phase, p.timeout_ns, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          // K step k: 8 more columns of the A slot, 32 more bytes of the
          // swizzled activation rows (+2 in the descriptor's address field)
          const uint32_t a_tmem = tmem_base + static_cast<uint32_t>(2 * BN + slot * 32);
          const uint64_t db0 = smem_desc_sw128(smem_addr(smem_x + stage * L::kXBytes));
#pragma unroll
          for (int k = 0; k < kBlockK / 16; ++k)
            tc_mma_f16_tmem_a(d_tmem, a_tmem + 8 * k, db0 + 2 * k, idesc,
                              (kb != 0 || k != 0) ? 1u : 0u);
          tc_commit(&empty_bar[stage]);
          tc_commit(&a_empty[slot]);
          if (++stage == Stages) {
            stage = 0;
            phase ^= 1;
          }
          if (++slot == kSlots) {
            slot = 0;
            a_phase ^= 1;
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
        tc_commit(drain_bar);
        mbar_wait(drain_bar, 0, p.timeout_ns, p.status);
      }
    }
  } else if (quarter >= 0) {
    // ------------------------------------------------------------ converters
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const int row = quarter * 32 + lane;  // this lane's weight row of the tile
    int stage = 0, slot = 0;
    uint32_t phase = 0, a_phase = 0;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      for (int kb = 0; kb < p.num_k_blocks; ++kb) {
        // the stage's codes have landed, and the slot's previous MMAs are done
        bool ready =
            mbar_wait_abortable(&w_full[stage], phase, p.timeout_ns, p.status, abort_flag) &&
            mbar_wait_abortable(&a_empty[slot], a_phase ^ 1, p.timeout_ns, p.status, abort_flag);
        if (!__all_sync(0xffffffffu, ready)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint4* src = reinterpret_cast<const uint4*>(smem_w + stage * L::kWBytes + row * 32);
        const uint4 c0 = src[0], c1 = src[1];
        const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        uint32_t f[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) e2m1x8_to_f16x2x4(words[i], f + 4 * i);
        tc::tmem_st_32cols(tmem_base + lane_addr + static_cast<uint32_t>(2 * BN + slot * 32), f);
        tc::tc_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[slot]);
        if (++stage == Stages) {
          stage = 0;
          phase ^= 1;
        }
        if (++slot == kSlots) {
          slot = 0;
          a_phase ^= 1;
        }
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    // Warps w and w + 4 share lane quarter w % 4 (32 weight rows = 32 columns
    // of D) and take alternate halves of the tile's 32-column chunks (32 rows
    // of D each).  Lane r holds D column n = 32 q + r of the tile; it writes
    // its 32 values down column r of a 32 x 32 box (rows of 64 bytes, so each
    // of the 32 stores of the warp covers one row, free of bank conflicts),
    // which TMA stores to D.  With beta != 0 TMA first brings C's box in.
    const int wi = warp - kEpiWarp0;
    const int q = wi & 3;
    const int half = wi >> 2;
    constexpr int kChunks = BN / 32;
    const int chunk_lo = half == 0 ? 0 : (kChunks + 1) / 2;
    const int chunk_hi = half == 0 ? (kChunks + 1) / 2 : kChunks;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    uint8_t* boxes = smem + L::kOffEpi + wi * 2 * kBoxBytes;
    uint64_t* cbar = epi_bar + wi * 2;
    const bool has_c = p.epi.beta != 0.0f;
    const bool has_bias = (p.epi.flags & kEpiBias) != 0;
    const uint64_t pol_c = policy_evict_first();
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t c_phase = 0;  // bit b: parity of box b's next C arrival
    int j = 0;             // boxes used so far (box j & 1 next)
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      int w_blk, x_blk;
      w4t_coords(p, t, w_blk, x_blk);
      const int n0 = w_blk * kBlockM + q * 32;  // D column of lane 0
      const int n = n0 + lane;
      const float b = (has_bias && n < p.N) ? __half2float(p.bias[n]) : 0.0f;
      const bool ready = !aborted(abort_flag) &&
                         mbar_wait_sleepy(&tmem_full[acc], acc_phase, p.timeout_ns, p.status, 256);
      if (!__all_sync(0xffffffffu, ready)) {
        *abort_flag = 1;
        ok = false;
        break;
      }
      tc_fence_after_sync();
#pragma unroll 1
      for (int c = chunk_lo; c < chunk_hi; ++c) {
        const int m0 = x_blk * BN + c * 32;  // D row of the chunk's first value
        const bool live = m0 < p.M && n0 < p.N;
        if (!live) continue;  // warp-uniform: the box lies wholly outside D
        uint32_t r[32];
        tmem_ld_32cols(tmem_base + lane_base + static_cast<uint32_t>(acc * BN + c * 32), r);
        const int bx = j & 1;
        uint8_t* box = boxes + bx * kBoxBytes;
        bool got = true;
        if (lane == 0) {
          bulk_wait_group_read<1>();  // the store that last read box bx has read it
          if (has_c) {
            mbar_arrive_expect_tx(&cbar[bx], kBoxBytes);
            tma_load_2d(&tmap_c, &cbar[bx], box, n0, m0, pol_c);
          }
        }
        __syncwarp();
        if (has_c) {
          got = mbar_wait(&cbar[bx], (c_phase >> bx) & 1u, p.timeout_ns, p.status);
          c_phase ^= 1u << bx;
        }
        got = __all_sync(0xffffffffu, got);
        tc_wait_ld();
        if (!got) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        __half* col = reinterpret_cast<__half*>(box) + lane;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float cv = has_c ? __half2float(col[i * 32]) : 0.0f;
          col[i * 32] = __float2half_rn(epi_apply(__uint_as_float(r[i]), cv, b, p.epi, prog));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmap_d, box, n0, m0);
          bulk_commit_group();
        }
        ++j;
      }
      if (!ok) break;
      tc_fence_before_sync();
      mbar_arrive(&tmem_empty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (lane == 0) bulk_wait_group<0>();  // stores end before the CTA does
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after_sync();
    tmem_dealloc<512>(tmem_base);
  }
}

template <int BN, int Stages>
int w4t_regs() {
  static std::atomic<int> slot{-1};
  return kernel_regs(gemm_w4t_kernel<BN, Stages>, slot);
}

template <int BN, int Stages>
cudaError_t run_w4t(const GemmArgs& a, const dg_tile_plan& plan) {
  using L = W4tSmem<BN, Stages>;
  CUtensorMap tx, tw, tcm, td;
  cudaError_t e = tc::make_f16_kmajor_map(&tx, a.A, a.M, a.K, a.lda, BN);
  if (e != cudaSuccess) return e;
  // codes as bytes: rows of ldb / 2 bytes, boxes of 32 bytes (64 values of
  // K) by 128 rows; the zero fill past the row gives code 0 (value 0)
  e = tc::make_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, a.N, (a.K + 1) / 2, a.ldb / 2,
                      kBlockM, kBlockK / 2, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  e = tc::make_map_2d(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.D, a.M, a.N, a.ldd * 2, 32, 32,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  tcm = td;
  if (a.beta != 0.0f) {
    e = tc::make_map_2d(&tcm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.C, a.M, a.N, a.ldc * 2, 32, 32,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  W4tParams p;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.num_w_blocks = static_cast<int>((a.N + kBlockM - 1) / kBlockM);
  p.num_x_blocks = static_cast<int>((a.M + BN - 1) / BN);
  p.num_tiles = p.num_w_blocks * p.num_x_blocks;
  p.num_k_blocks = static_cast<int>((a.K + kBlockK - 1) / kBlockK);
  p.epi = make_epi(a);
  p.bias = static_cast<const __half*>(a.bias);
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;

  auto kern = gemm_w4t_kernel<BN, Stages>;
  int dev = 0;
  cudaGetDevice(&dev);
  static std::atomic<uint64_t> attr_set{0};
  e = once_per_device(attr_set, dev, [&]() {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                L::kLaunchBytes);
  });
  if (e != cudaSuccess) return e;
  int grid = plan.grid > 0 ? plan.grid : a.sm_count;
  if (grid > p.num_tiles) grid = p.num_tiles;
  if (grid < 1) grid = 1;
  e = launch_dependent(kern, dim3(grid), dim3(kThreads), L::kLaunchBytes, a.stream, tx, tw, tcm,
                       td, p, make_program(a));
  count_launches(1);
  return e;
}

}  // namespace

// Layouts the kernel reads and writes with TMA: 16-byte aligned bases, rows
// of A a multiple of 8 values, rows of codes a multiple of 16 bytes, rows of
// D (and of C when read) a multiple of 8 values; FP16 output.
bool w4t_layout_ok(const GemmArgs& a) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (a.dtype_a != DG_F16 || a.dtype_b != DG_E2M1 || (a.epi & kEpiOutI8)) return false;
  if (!al16(a.A) || a.lda % 8 != 0 || !al16(a.B) || a.ldb % 32 != 0) return false;
  if (!al16(a.D) || a.ldd % 8 != 0) return false;
  if (a.beta != 0.0f && (!al16(a.C) || a.ldc % 8 != 0)) return false;
  return true;
}

int w4t_kernel_regs(int n_tile, int stages) {
  if (n_tile == 160 && stages == 7) return w4t_regs<160, 7>();
  if (n_tile == 224 && stages == 6) return w4t_regs<224, 6>();
  return 0;
}

// FP16 activations x packed E2M1 weights, D^T tiles of 128 weight rows x
// plan.n_tile activation rows (plan.swap_ab == 1).
cudaError_t launch_w4t(const GemmArgs& a, const dg_tile_plan& plan) {
  // 160 rows: six A slots; 224 rows: two, but 448 cycles of MMA a stage,
  // half again the converters' time
  if (plan.n_tile == 160 && plan.stages == 7) return run_w4t<160, 7>(a, plan);
  if (plan.n_tile == 224 && plan.stages == 6) return run_w4t<224, 6>(a, plan);
  return cudaErrorNotSupported;
}

}  // namespace dg
