// Tensor-core GEMM for operands that are not FP16 in memory: INT8 x INT8 with
// an exact INT32 result, and FP16 activations x packed 4-bit E2M1 weights
// (W4A16) with the fused FP16 epilogue.
//
// Sources: INT8 4096^3 GEMM with INT32 output (discosf.com/news/5532976,
// section 1 and section 4.3); the {weight: int4_e2m1, activation: fp16,
// output: fp16} precision triple with 2 exponent + 1 mantissa bits (same
// article, section 2.2 layer 2) packed two codes per byte (section 4.3,
// "pack_int4"); bias + GELU fused (kwkr.cn/news/562171, section 2.2 third
// layer).
//
// sm_103a has no integer tcgen05.mma and no mixed FP16 x FP4 kind, and its
// legacy mma.sync s8 path is slow, so both contractions run on the FP16
// tensor-core path with the narrow operand widened in shared memory:
//
//   warp 0       TMA producer into a deep input ring (`SIn` slots): raw int8
//                / packed-E2M1 tiles (no swizzle) and FP16 A tiles (128-byte
//                swizzle);
//   warps 8-11   converters: raw -> FP16 in the swizzled K-major layout the
//                MMA reads, into a short converted ring (`SCv` slots) (int8:
//                exact via the 1024+u magic-number trick; E2M1:
//                cvt.rn.f16x2.e2m1x2, exact), then a proxy fence;
//   warp 1       MMA issuer: tcgen05.mma kind::f16 into TMEM (FP32); its
//                commits free both the input and the converted slot;
//   warp 2       TMEM allocation;  warps 4-7  epilogue.
// The input ring is deep because it must cover the TMA latency; the wide
// converted tiles need only cover the conversion latency.
//
// INT8 exactness: every product is an integer of magnitude <= 2^14, so any
// partial sum of at most 1024 products is an integer of magnitude <= 2^24 and
// exact in FP32.  The MMA therefore accumulates K in chunks of 1024 into one
// of two FP32 TMEM buffers; the epilogue converts each finished chunk to INT32
// (exact) and adds it into an INT32 running sum kept in a third TMEM region.
// The last chunk produces D = alpha*sum + beta*C in INT32 (wrapping mod 2^32).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "convert.cuh"
#include "tc_common.cuh"

namespace dg {
namespace {

using tc::kBlockK;
using tc::kBlockM;

enum : int { kOpF16 = 0, kOpI8 = 1, kOpE2M1 = 2 };
enum : int { kOutF16 = 0, kOutI32 = 1 };

constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kConvWarp0 = 8;
constexpr int kConvThreads = 128;
using tc::kI32ChunkKb;

struct ConvParams {
  int M, N, K;
  int num_m_blocks, num_n_blocks, num_tiles, num_k_blocks;
  int group_m;
  Epi epi;
  const void* C;  // read when beta != 0 (FP16, or INT32 when Out == kOutI32)
  int64_t ldc;
  void* D;
  int64_t ldd;
  const __half* bias;
  int32_t alpha_i, beta_i;
  int* status;
  uint64_t timeout_ns;
  uint32_t stage_tx;  // bytes TMA delivers per input slot
};
static_assert(sizeof(ConvParams) <= 128, "parameter struct within 128 bytes (see Epi)");

template <int BN, int SIn, int SCv, int OpA, int OpB>
struct ConvSmem {
  // input slot: A as loaded (FP16 tile or raw int8), B raw
  static constexpr int kInA = OpA == kOpF16 ? kBlockM * kBlockK * 2 : kBlockM * kBlockK;
  static constexpr int kInB = OpB == kOpI8 ? BN * kBlockK : BN * kBlockK / 2;
  // converted slot: widened A (when A is not FP16) and widened B
  static constexpr int kCvA = OpA == kOpF16 ? 0 : kBlockM * kBlockK * 2;
  static constexpr int kCvB = BN * kBlockK * 2;
  static constexpr int kOffInA = 0;
  static constexpr int kOffInB = kOffInA + SIn * kInA;
  static constexpr int kOffCvA = kOffInB + SIn * kInB;
  static constexpr int kOffCvB = kOffCvA + SCv * kCvA;
  static constexpr int kOffBar = kOffCvB + SCv * kCvB;
  // in_full[SIn], in_empty[SIn], cv_full[SCv], cv_empty[SCv], tmem_full[2], tmem_empty[2], drain
  static constexpr int kNumBars = 2 * SIn + 2 * SCv + 5;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kBytes = kOffAbort + 4;
  static constexpr int kLaunchBytes = kBytes + 1024;
  static_assert(kInA % 1024 == 0 && kInB % 1024 == 0 && kCvA % 1024 == 0 && kCvB % 1024 == 0,
                "tiles keep 1 KB alignment");
  static_assert(kLaunchBytes <= 232448, "shared memory per CTA");
};

__device__ __forceinline__ bool aborted(volatile int* flag) { return *flag != 0; }

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Four int8 (one 32-bit word) -> four FP16 (two 32-bit words), exact:
// byte b -> fp16 bits 0x6400 | (b ^ 0x80) = 1024 + (v + 128), minus 1152.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;
  uint32_t a = __byte_perm(x, 0x64646464u, 0x4140);
  uint32_t b = __byte_perm(x, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

// Byte offset of the 16-byte chunk c (0..7) of row r in a 128-byte-swizzled
// K-major tile (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B).
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// Widen one slot's raw tile of `Rows` rows into the FP16 operand tile.
// Thread ct owns output chunk c = ct % 8 of rows ct / 8 + 16 i: its chunk and
// swizzle phase (row % 8) are the same in every iteration, so each step is
// one load, the conversion and one store at fixed strides.
template <int Op, int Rows>
__device__ __forceinline__ void convert_tile(const uint8_t* raw, uint8_t* op, int ct) {
  constexpr int kRowsPerStep = kConvThreads / 8;  // 16
  constexpr int kRawRow = Op == kOpI8 ? 64 : 32;  // raw bytes per row
  constexpr int kRawChunk = Op == kOpI8 ? 8 : 4;  // raw bytes per output chunk
  const int r0 = ct >> 3, c = ct & 7;
  const uint8_t* src = raw + r0 * kRawRow + c * kRawChunk;
  uint8_t* dst = op + sw128_offset(r0, c);  // (r0 + 16 i) % 8 == r0 % 8
#pragma unroll
  for (int i = 0; i < Rows / kRowsPerStep; ++i) {
    uint4 o;
    if (Op == kOpI8) {
      const uint2 w = *reinterpret_cast<const uint2*>(src + i * kRowsPerStep * kRawRow);
      i8x4_to_f16x4(w.x, o.x, o.y);
      i8x4_to_f16x4(w.y, o.z, o.w);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(src + i * kRowsPerStep * kRawRow);
      o = e2m1x8_to_f16x8(w);
    }
    *reinterpret_cast<uint4*>(dst + i * kRowsPerStep * 128) = o;
  }
}

// Position in the two rings of the i-th K block this CTA processes.
struct RingPos {
  int in, cv;
  uint32_t in_phase, cv_phase;
  __device__ __forceinline__ RingPos() : in(0), cv(0), in_phase(0), cv_phase(0) {}
  template <int SIn, int SCv>
  __device__ __forceinline__ void advance() {
    if (++in == SIn) {
      in = 0;
      in_phase ^= 1;
    }
    if (++cv == SCv) {
      cv = 0;
      cv_phase ^= 1;
    }
  }
};

template <int BN, int SIn, int SCv, int OpA, int OpB, int Out>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_conv_tc_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b, const ConvParams p,
                        const __grid_constant__ EpiProgram prog) {
  using L = ConvSmem<BN, SIn, SCv, OpA, OpB>;
  constexpr bool kConvA = OpA != kOpF16;
  static_assert(OpB != kOpF16, "B is always the widened operand here");
  // FP32 accumulators x2, plus the INT32 running sums on the integer path.
  constexpr int kColsNeeded = Out == kOutI32 ? 3 * BN : 2 * BN;
  constexpr int kTmemCols = kColsNeeded <= 128 ? 128 : (kColsNeeded <= 256 ? 256 : 512);
  constexpr uint32_t kIdesc = idesc_f16_f32(kBlockM, BN);
  static_assert(kColsNeeded <= 512, "tensor memory");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* in_full = bars;
  uint64_t* in_empty = bars + SIn;
  uint64_t* cv_full = bars + 2 * SIn;
  uint64_t* cv_empty = bars + 2 * SIn + SCv;
  uint64_t* tmem_full = bars + 2 * SIn + 2 * SCv;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* drain_bar = tmem_full + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // K blocks per accumulation chunk (one FP32 accumulator fill).
  const int chunk_kb = Out == kOutI32 ? kI32ChunkKb : p.num_k_blocks;
  const int num_chunks = (p.num_k_blocks + chunk_kb - 1) / chunk_kb;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SIn; ++s) {
      mbar_init(&in_full[s], 1);
      mbar_init(&in_empty[s], 1);
    }
    for (int s = 0; s < SCv; ++s) {
      mbar_init(&cv_full[s], kConvThreads);
      mbar_init(&cv_empty[s], 1);
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
  // Launched as a dependent of the previous kernel in the stream: the set-up
  // above touched only on-chip state; global memory waits for that kernel.
  grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one_lane()) {
      // operand tiles are read again by other tiles: they outrank C and D in L2
      const uint64_t pol = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        int m_blk, n_blk;
        tc::tile_coords(t, p.num_m_blocks, p.num_n_blocks, p.group_m, m_blk, n_blk);
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          if (aborted(abort_flag) ||
              !mbar_wait(&in_empty[stage], phase ^ 1, p.timeout_ns, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&in_full[stage], p.stage_tx);
          tma_load_2d(&tmap_a, &in_full[stage], smem + L::kOffInA + stage * L::kInA,
                      kb * kBlockK, m_blk * kBlockM, pol);
          // int8 rows carry 64 bytes per K block, packed E2M1 rows 32
          tma_load_2d(&tmap_b, &in_full[stage], smem + L::kOffInB + stage * L::kInB,
                      OpB == kOpI8 ? kb * kBlockK : kb * (kBlockK / 2), n_blk * BN, pol);
          ++issued;
          if (++stage == SIn) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Every operand load is issued: a kernel launched after this one may be
      // scheduled now (not earlier: its blocks could wait beside this CTA).
      grid_launch_dependents();
      if (!ok) {
        *abort_flag = 1;
        const int64_t first = issued > SIn ? issued - SIn : 0;
        for (int64_t i = first; i < issued; ++i)
          mbar_wait(&in_full[i % SIn], static_cast<uint32_t>((i / SIn) & 1), p.timeout_ns,
                    p.status);
      }
    }
  } else if (warp >= kConvWarp0) {
    // ------------------------------------------------------------ converters
    const int ct = threadIdx.x - kConvWarp0 * 32;
    RingPos pos;
    bool ok = true;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      for (int kb = 0; kb < p.num_k_blocks; ++kb) {
        if (aborted(abort_flag) ||
            !mbar_wait(&in_full[pos.in], pos.in_phase, p.timeout_ns, p.status) ||
            !mbar_wait(&cv_empty[pos.cv], pos.cv_phase ^ 1, p.timeout_ns, p.status)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        if (kConvA)
          convert_tile<OpA, kBlockM>(smem + L::kOffInA + pos.in * L::kInA,
                                     smem + L::kOffCvA + pos.cv * L::kCvA, ct);
        convert_tile<OpB, BN>(smem + L::kOffInB + pos.in * L::kInB,
                              smem + L::kOffCvB + pos.cv * L::kCvB, ct);
        fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
        mbar_arrive(&cv_full[pos.cv]);
        pos.advance<SIn, SCv>();
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one_lane()) {
      RingPos pos;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        for (int ch = 0; ch < num_chunks && ok; ++ch) {
          if (aborted(abort_flag) ||
              !mbar_wait(&tmem_empty[acc], acc_phase ^ 1, p.timeout_ns, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
          const int kb0 = ch * chunk_kb;
          const int kb1 = min(p.num_k_blocks, kb0 + chunk_kb);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (aborted(abort_flag) ||
                !mbar_wait(&in_full[pos.in], pos.in_phase, p.timeout_ns, p.status) ||
                !mbar_wait(&cv_full[pos.cv], pos.cv_phase, p.timeout_ns, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t a0 = smem_addr(kConvA ? smem + L::kOffCvA + pos.cv * L::kCvA
                                                 : smem + L::kOffInA + pos.in * L::kInA);
            const uint32_t b0 = smem_addr(smem + L::kOffCvB + pos.cv * L::kCvB);
#pragma unroll
            for (int k = 0; k < kBlockK / 16; ++k) {
              tc_mma_f16(d_tmem, smem_desc_sw128(a0 + k * 32), smem_desc_sw128(b0 + k * 32),
                         kIdesc, (kb != kb0 || k != 0) ? 1u : 0u);
            }
            tc_commit(&in_empty[pos.in]);
            tc_commit(&cv_empty[pos.cv]);
            pos.advance<SIn, SCv>();
          }
          if (!ok) break;
          tc_commit(&tmem_full[acc]);
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        tc_commit(drain_bar);
        mbar_wait(drain_bar, 0, p.timeout_ns, p.status);
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - kEpiWarp0;
    const uint32_t lane_base = static_cast<uint32_t>(ew * 32) << 16;
    const uint32_t sums = tmem_base + lane_base + 2 * BN;  // INT32 running sums
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      int m_blk, n_blk;
      tc::tile_coords(t, p.num_m_blocks, p.num_n_blocks, p.group_m, m_blk, n_blk);
      const int row = m_blk * kBlockM + ew * 32 + lane;
      for (int ch = 0; ch < num_chunks; ++ch) {
        if (aborted(abort_flag) ||
            !mbar_wait_sleepy(&tmem_full[acc], acc_phase, p.timeout_ns, p.status, 256)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t tacc = tmem_base + lane_base + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32cols(tacc + c * 32, r);
          tc_wait_ld();
          const int col0 = n_blk * BN + c * 32;
          if (Out == kOutF16) {
            if (col0 < p.N)
              tc::epilogue_f16_chunk(r, row, col0, p.M, p.N, p.epi, prog,
                                     static_cast<const __half*>(p.C), p.ldc,
                                     static_cast<__half*>(p.D), p.ldd, p.bias);
          } else {
            tc::flush_i32_piece(r, sums + c * 32, ch == 0, ch + 1 == num_chunks, row, col0, p.M,
                                p.N, p.alpha_i, p.beta_i,
                                tc::I32Out{static_cast<const int32_t*>(p.C), p.ldc,
                                           static_cast<int32_t*>(p.D), p.ldd});
          }
        }
        tc_fence_before_sync();
        mbar_arrive(&tmem_empty[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
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

template <int BN, int SIn, int SCv, int OpA, int OpB, int Out>
cudaError_t run_conv(const GemmArgs& a, const dg_tile_plan& plan) {
  using L = ConvSmem<BN, SIn, SCv, OpA, OpB>;
  // Fewer than 128 rows: load only those rows (rounded up to 8); the stale
  // shared-memory rows below only feed accumulator rows >= M.
  const int box_a = a.M < kBlockM ? static_cast<int>((a.M + 7) / 8 * 8) : kBlockM;
  CUtensorMap ta, tb;
  cudaError_t e;
  if (OpA == kOpF16)
    e = tc::make_f16_kmajor_map(&ta, a.A, a.M, a.K, a.lda, box_a);
  else  // int8: rows of K bytes, 64-byte boxes, no swizzle
    e = tc::make_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.A, a.M, a.K, a.lda, box_a, kBlockK,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  if (OpB == kOpI8)
    e = tc::make_map_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, a.N, a.K, a.ldb, BN, kBlockK,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
  else  // E2M1: rows of ceil(K/2) bytes, pitch ldb/2 bytes, 32-byte boxes
    e = tc::make_map_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, a.N, (a.K + 1) / 2, a.ldb / 2,
                        BN, kBlockK / 2, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;

  ConvParams p;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.num_m_blocks = static_cast<int>((a.M + kBlockM - 1) / kBlockM);
  p.num_n_blocks = static_cast<int>((a.N + BN - 1) / BN);
  p.num_tiles = p.num_m_blocks * p.num_n_blocks;
  p.num_k_blocks = static_cast<int>((a.K + kBlockK - 1) / kBlockK);
  p.group_m = 16;
  p.epi = make_epi(a);
  p.C = a.C;
  p.ldc = a.ldc;
  p.D = a.D;
  p.ldd = a.ldd;
  p.bias = static_cast<const __half*>(a.bias);
  p.alpha_i = static_cast<int32_t>(a.alpha);
  p.beta_i = static_cast<int32_t>(a.beta);
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  p.stage_tx = static_cast<uint32_t>(box_a * (OpA == kOpF16 ? kBlockK * 2 : kBlockK) + L::kInB);

  auto kern = gemm_conv_tc_kernel<BN, SIn, SCv, OpA, OpB, Out>;
  int dev = 0;
  cudaGetDevice(&dev);
  static std::atomic<uint64_t> attr_set{0};  // one shared-memory opt-in per variant and device
  e = once_per_device(attr_set, dev, [&]() {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                L::kLaunchBytes);
  });
  if (e != cudaSuccess) return e;
  int grid = plan.grid > 0 ? plan.grid : a.sm_count;
  if (grid > p.num_tiles) grid = p.num_tiles;
  e = launch_dependent(kern, dim3(grid), dim3(kThreads), L::kLaunchBytes, a.stream, ta, tb, p,
                       make_program(a));
  count_launches(1);
  return e;
}

}  // namespace

// Shapes compiled for the converting kernels; the planner proposes only these.
// (N_tile, input slots, converted slots) per dtype pair.
namespace {
template <int BN, int Stages, int CvStages, int OpA, int OpB, int Out>
int conv_regs_of() {
  static std::atomic<int> slot{-1};
  return kernel_regs(gemm_conv_tc_kernel<BN, Stages, CvStages, OpA, OpB, Out>, slot);
}
}  // namespace

int conv_kernel_regs(dg_dtype da, dg_dtype db, int n_tile, int stages) {
  if (da == DG_I8 && db == DG_I8) {
    if (n_tile == 128 && stages == 8) return conv_regs_of<128, 8, 3, kOpI8, kOpI8, kOutI32>();
  } else if (da == DG_F16 && db == DG_E2M1) {
    if (n_tile == 256 && stages == 6) return conv_regs_of<256, 6, 2, kOpF16, kOpE2M1, kOutF16>();
    if (n_tile == 128 && stages == 8) return conv_regs_of<128, 8, 3, kOpF16, kOpE2M1, kOutF16>();
    if (n_tile == 64 && stages == 8) return conv_regs_of<64, 8, 4, kOpF16, kOpE2M1, kOutF16>();
  }
  return 0;
}

cudaError_t launch_conv(const GemmArgs& a, const dg_tile_plan& plan) {
  if (a.dtype_a == DG_I8 && a.dtype_b == DG_I8) {
    if (plan.n_tile == 128 && plan.stages == 8)
      return run_conv<128, 8, 3, kOpI8, kOpI8, kOutI32>(a, plan);
  } else if (a.dtype_a == DG_F16 && a.dtype_b == DG_E2M1) {
    if (plan.n_tile == 256 && plan.stages == 6)
      return run_conv<256, 6, 2, kOpF16, kOpE2M1, kOutF16>(a, plan);
    if (plan.n_tile == 128 && plan.stages == 8)
      return run_conv<128, 8, 3, kOpF16, kOpE2M1, kOutF16>(a, plan);
    if (plan.n_tile == 64 && plan.stages == 8)
      return run_conv<64, 8, 4, kOpF16, kOpE2M1, kOutF16>(a, plan);
  }
  return cudaErrorNotSupported;
}

}  // namespace dg
