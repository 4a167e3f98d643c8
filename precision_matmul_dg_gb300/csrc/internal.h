// Declarations shared by the host translation units of libdg (not exported).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <string>
#include <utility>

#include "dg.h"

namespace dg {

// Epilogue flags as the kernels see them.
// kEpiOutI8: the program ends in an int8 quantization and D is int8.
enum : int { kEpiBias = 1, kEpiGelu = 2, kEpiProgram = 4, kEpiOutI8 = 8 };

// Epilogue-program ops (dg_epilogue_op of dg.h).
using EpiOp = dg_epilogue_op;
constexpr int kMaxEpiOps = DG_MAX_EPILOGUE_OPS;
enum : int {
  kOpBias = DG_OP_BIAS,
  kOpRelu = DG_OP_RELU,
  kOpGelu = DG_OP_GELU,
  kOpScale = DG_OP_SCALE,
  kOpClamp = DG_OP_CLAMP,
  kOpQuantI8 = DG_OP_QUANT_I8
};

// Launches `kern` with programmatic stream serialization: its CTAs may be
// scheduled (and run their set-up) while the previous kernel in the stream
// drains.  Every kernel launched this way executes griddepcontrol.wait
// before its first global-memory access, which waits for that kernel to
// complete and its memory to be visible.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// One-time set-up of a kernel on a device (shared-memory opt-in, occupancy
// query), safe when several host threads make their first call at once:
// `init` runs under a lock, at most once per device and flag word (retried
// after a failure), and what it wrote is visible to every later caller that
// finds the device's bit set.
template <typename F>
cudaError_t once_per_device(std::atomic<uint64_t>& done, int dev, F&& init) {
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (done.load(std::memory_order_relaxed) & bit) return cudaSuccess;
  const cudaError_t e = init();
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Registers per thread that ptxas gave `kern`, read once with
// cudaFuncGetAttributes and kept in `slot` (which starts at -1).  0 when no
// device is present to read them from; the planner then uses its bound.
template <typename Kern>
int kernel_regs(Kern kern, std::atomic<int>& slot) {
  int v = slot.load(std::memory_order_acquire);
  if (v >= 0) return v;
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(kern)) == cudaSuccess) {
    v = fa.numRegs;
  } else {
    cudaGetLastError();
    v = 0;
  }
  slot.store(v, std::memory_order_release);
  return v;
}

// Everything a launcher needs to run one GEMM, already validated.
struct GemmArgs {
  int64_t M, N, K;
  dg_dtype dtype_a, dtype_b;
  const void* A;
  int64_t lda;
  const void* B;
  int64_t ldb;
  const void* C;  // read when beta != 0; else equal to D
  int64_t ldc;    // row pitches in elements (N for dg_gemm, where C == D)
  void* D;        // C and D are one buffer (ldc == ldd) or do not overlap
  int64_t ldd;
  const void* bias;
  float alpha, beta;
  int epi;    // kEpiBias | kEpiGelu, or kEpiProgram (+ kEpiBias)
  int n_ops;  // kEpiProgram: the ops, in order
  EpiOp ops[kMaxEpiOps];
  // Strided batch (GEMV kernel only): `batch` problems, problem z at
  // A + z stride_a, B + z stride_b, C + z stride_c, D + z stride_d,
  // bias + z stride_bias (elements).  1 for a single problem.
  int64_t batch;
  int64_t stride_a, stride_b, stride_c, stride_d, stride_bias;
  cudaStream_t stream;
  int* status;          // per-device status word (device memory)
  uint64_t timeout_ns;  // device-side wait limit
  int sm_count;
  bool exact_i32;       // FP16 operands hold widened INT8 values: exact INT32 output
  bool bf16_ab = false;  // A and B are BF16 (widened MXFP4 operands), not FP16
  // MXFP4 operands (dtype DG_MXF4): E8M0 scale bytes, row pitches in bytes
  const void* scale_a = nullptr;
  int64_t lds_a = 0;
  const void* scale_b = nullptr;
  int64_t lds_b = 0;
};

// Measured registers per thread of the kernel a plan would launch (0 when
// they cannot be read: no device).  FP16 tensor-core kernel (gemm_tc.cu;
// exact_i32: its INT32 output mode), converting kernel (gemm_conv.cu),
// split-K GEMV and warp-MMA GEMV for M rows (gemv.cu), skinny W4A16 kernel
// (skinny.cu).  0 too for a variant that is not compiled.
int tc_kernel_regs(int n_tile, int stages, int cta_group, bool exact_i32);
int tc_streamk_kernel_regs(int n_tile, int stages, int cta_group);  // stream-K (gemm_tc.cu)
int mx_kernel_regs(int n_tile, int stages, int cta_group);  // MXFP4 block-scaled (gemm_tc.cu)
int conv_kernel_regs(dg_dtype da, dg_dtype db, int n_tile, int stages);
int gemv_kernel_regs(int64_t M, int split);
int gemv_mma_kernel_regs(int64_t M);
int skinny_kernel_regs();

// Planner (planner.cpp) -- host only.
dg_status plan_tiles(int64_t M, int64_t N, int64_t K, dg_dtype dtype_a, dg_dtype dtype_b,
                     dg_epilogue epilogue, const dg_hw_desc& hw, double target_occupancy,
                     dg_tile_plan* out, int max_out, int* n_out, std::string* why);

// Whether the kernels shipped here can run `plan` for this problem.
bool plan_is_runnable(const dg_tile_plan& plan, int64_t M, int64_t N, int64_t K,
                      dg_dtype dtype_a, dg_dtype dtype_b, std::string* why);

// Scratch for split-K reductions: FP32 partial sums and arrival counters.
struct SplitKWorkspace {
  float* partial;
  int64_t partial_elems;
  unsigned* counters;
  int64_t counter_elems;
};

// Stream-K division of `tiles` output tiles of `kblocks` K blocks each over
// `units` scheduling units (CTAs, or CTA pairs), as the stream-K kernel
// walks it: tiles [0, dp_tiles) whole, then the sk_iters K blocks of the
// other sk_tiles tiles cut into sk_units contiguous ranges of equal length
// (+-1); a tile meets at most max_pieces ranges.  With fewer tiles than
// units every tile is cut into the same number of equal ranges.
// sk_tiles == 0: the tiles fill whole waves, a tile has one K block, or
// fewer tiles than units leave no two units per tile: nothing to balance.
// Host only (planner.cpp).
struct SkSplit {
  int64_t dp_tiles, sk_tiles, sk_iters;
  int sk_units, max_pieces;
};
SkSplit stream_k_split(int64_t tiles, int64_t kblocks, int64_t units);

// Scratch of the stream-K kernel on (device, stream) (api.cu): at least
// `partial_elems` FP32 partial sums, and `sync_elems` words (the launch
// epoch, a count of finished CTAs, then the flags) zeroed when allocated.
dg_status get_sk_workspace(int dev, cudaStream_t stream, int64_t partial_elems,
                           int64_t sync_elems, float** partial, unsigned** sync);

// Launchers (gemm_tc.cu, gemv.cu).  Each returns cudaSuccess or the launch error.
cudaError_t launch_tc(const GemmArgs& a, const dg_tile_plan& plan);    // F16 x F16
// F16 x F16 with stream-K work division (DG_KERNEL_TC_STREAMK plans).
cudaError_t launch_tc_streamk(const GemmArgs& a, const dg_tile_plan& plan);
// F16 x E2M1 with the weights widened in tensor memory (gemm_w4t.cu):
// DG_KERNEL_TC plans with swap_ab == 1 (tiles of 128 weight rows x n_tile
// activation rows).  w4t_layout_ok: the operand and output layouts its TMA
// copies need (otherwise the call runs the widening path).
cudaError_t launch_w4t(const GemmArgs& a, const dg_tile_plan& plan);
bool w4t_layout_ok(const GemmArgs& a);
int w4t_kernel_regs(int n_tile, int stages);
// MXFP4 x MXFP4 on the block-scaled MMA (gemm_tc.cu): a.A, a.B packed codes
// with K even; a.scale_a, a.scale_b 16-byte aligned with lds_a, lds_b
// multiples of 16.
cudaError_t launch_tc_mx(const GemmArgs& a, const dg_tile_plan& plan);
cudaError_t launch_conv(const GemmArgs& a, const dg_tile_plan& plan);  // I8 x I8, F16 x E2M1
cudaError_t launch_gemv(const GemmArgs& a, const dg_tile_plan& plan, const SplitKWorkspace& ws);
// Warp-MMA GEMV (gemv.cu): F16 x F16 with M <= 16 on m16n8k16 tensor-core MMAs.
cudaError_t launch_gemv_mma(const GemmArgs& a, const dg_tile_plan& plan,
                            const SplitKWorkspace& ws);
// The same over a group of problems of one N and K (dg_gemm_grouped): `table`
// is a device array of `count` entries written by gemv_group_entry, max_m the
// largest M.  a.N, a.K, a.lda, a.ldb, the epilogue and the stream apply to all.
cudaError_t launch_gemv_mma_grouped(const GemmArgs& a, const void* table, int64_t count,
                                    int64_t max_m, const dg_tile_plan& plan,
                                    const SplitKWorkspace& ws);
int64_t gemv_group_entry_bytes();
void gemv_group_entry(void* table, int64_t i, const void* A, const void* B, void* CD,
                      const void* bias, int64_t M);
// Skinny W4A16 kernel (skinny.cu): FP16 A with M <= 16 x packed E2M1 B.
cudaError_t launch_skinny(const GemmArgs& a, const dg_tile_plan& plan);
int skinny_smem_bytes();
int skinny_threads();
int skinny_cols_per_block();
int skinny_k_chunk();
cudaError_t launch_epilogue_only(const GemmArgs& a);

// Widening pre-pass (widen.cu): int8 or packed-E2M1 rows -> FP16 rows with
// leading dimension widened_ld(K).  One or two operands (A and B of an INT8
// product) per call, in one launch when both are dense and of one type.
int64_t widened_ld(int64_t K);
struct WidenJob {
  dg_dtype dtype;
  const void* src;
  int64_t rows, ld_src;  // ld_src in elements (codes for E2M1)
  __half* dst;
};
cudaError_t launch_widen(const WidenJob* jobs, int njobs, int64_t K, cudaStream_t stream,
                         int sm_count);
// MXFP4 (mx.cu): block quantization of FP16 rows (ldq in codes), and the
// exact widening of MXFP4 rows (codes + E8M0 scales) to BF16 rows of
// widened_ld(K) values, one or two operands per launch.
cudaError_t launch_quantize_mxf4(int64_t rows, int64_t K, const void* X, int64_t ldx,
                                 void* codes, int64_t ldq, void* scales, int64_t lds,
                                 cudaStream_t stream, int sm_count);
struct MxWidenJob {
  const void* codes;
  int64_t rows, ld;  // ld in codes (a multiple of 32)
  const void* scales;
  int64_t lds;       // bytes
  __half* dst;       // holds BF16 bits
};
cudaError_t launch_widen_mxf4(const MxWidenJob* jobs, int njobs, int64_t K, cudaStream_t stream,
                              int sm_count);
cudaError_t launch_wait_selftest(cudaStream_t stream, int* status, uint64_t timeout_ns);

// Whether the split-K GEMV reduces `split` splits inside a thread-block
// cluster (no workspace) rather than through global partial sums.
bool gemv_split_in_cluster(int split);
// Workspace sizes a GEMV plan needs for `batch` problems.
int64_t gemv_partial_elems(const dg_tile_plan& plan, int64_t M, int64_t N, int64_t batch);
int64_t gemv_counter_elems(const dg_tile_plan& plan, int64_t N, int64_t batch);

// Kernel-launch counter and error state (api.cu).  None of these allocate.
void count_launches(int n);
void clear_error();
dg_status set_error(dg_status s, const char* msg);
dg_status fill_hw_desc(int device, dg_hw_desc* out);
dg_status validate_gemm_args(int64_t M, int64_t N, int64_t K, dg_dtype da, dg_dtype db,
                             const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                             const void* bias, float alpha, float beta, dg_epilogue epi);

// Split-K choice of the GEMV kernel (planner.cpp): cost-model time of one
// split count (negative when the split is not allowed), and the best split.
// `batch` independent problems of the shape share one launch.
double gemv_estimate_us(int64_t M, int64_t N, int64_t K, int split, const dg_hw_desc& hw,
                        int64_t* chunk_out, int64_t batch = 1);
int gemv_best_split(int64_t M, int64_t N, int64_t K, const dg_hw_desc& hw, int64_t* chunk_out,
                    int64_t batch = 1);
// The same for the warp-MMA GEMV (2 <= M <= 16).
double gemv_mma_estimate_us(int64_t M, int64_t N, int64_t K, int split, const dg_hw_desc& hw,
                            int64_t* chunk_out, int64_t batch = 1);
int gemv_mma_best_split(int64_t M, int64_t N, int64_t K, const dg_hw_desc& hw,
                        int64_t* chunk_out, int64_t batch = 1);

}  // namespace dg
