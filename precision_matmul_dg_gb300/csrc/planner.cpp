// Tile planner: the constraint system of the "DeepGEMM" articles' first layer
// (kwkr.cn/news/562171, section 2.2, "Hardware-Aware Tile Planner"):
//
//   SharedMemoryUsage(M_tile, N_tile, K_tile, dtype) <= available shared memory
//   RegisterUsage(M_tile, N_tile, K_tile, dtype)     <= registers available
//   Occupancy(M_tile, N_tile, K_tile)                >= target (e.g. 0.7)
//
// solved for one hardware description and one problem, returning the
// surviving (M_tile, N_tile, K_tile, split-K, stages) candidates ranked by a
// cost model (section 3.2 step 2 of the same article; discosf.com/news/5532976
// section 4.1 stage 2 prunes an enumerated candidate space the same way).
//
// Two tile families are enumerated:
//  * Blackwell (hw.tmem_cols > 0): the kernels compiled into this library --
//    the tcgen05 tensor-core kernel (constraints add tensor-memory columns:
//    two 128 x N_tile FP32 accumulators) and the split-K GEMV for thin M.
//    These kernels are persistent with one CTA per SM by design, so
//    "occupancy" is read as wave efficiency: work units / (waves * SMs).
//  * Earlier GPUs (hw.tmem_cols == 0): a warp-level-MMA family in the pages'
//    own ranges (M, N in [16, 128], K in [16, 64]) with warp occupancy
//    (resident warps / maximum warps).  Planning only: this library has no
//    kernel for it, and dg_gemm_planned rejects such plans.
#include <math.h>

#include <algorithm>
#include <string>
#include <vector>

#include "internal.h"

namespace dg {
namespace {

// Shapes of the tcgen05 kernels compiled into gemm_tc.cu (FP16 x FP16) and
// gemm_conv.cu (INT8 x INT8, FP16 x E2M1): (N_tile, stages) per dtype pair.
// `stages` is the TMA ring depth; the converting kernel adds a ring of
// `cv_stages` widened-operand slots.
struct TcVariant {
  int n_tile, stages, cta_group, cv_stages;
};
constexpr TcVariant kTcVariantsF16[] = {{256, 4, 1, 0}, {128, 6, 1, 0}, {64, 8, 1, 0},
                                        {256, 6, 2, 0}, {224, 6, 2, 0}, {192, 6, 2, 0},
                                        {128, 8, 2, 0}};
constexpr int kNumTcVariantsF16 = 7;
// FP16 x E2M1 with the weights widened in tensor memory (gemm_w4t.cu): D^T
// tiles of 128 weight rows x n_tile activation rows, single CTAs, 448
// threads; shared memory: per stage an activation tile (n_tile rows of 128
// bytes) and 4 KB of codes, and 32 KB of epilogue boxes
constexpr TcVariant kW4tVariants[] = {{160, 7, 1, 0}, {224, 6, 1, 0}};
constexpr int kW4tThreads = 448;
// Its cost per tile: a fixed part and the stages at this fraction of the
// tensor rate (the converters widen every weight again for each activation
// tile and share the SMs' issue slots with the epilogue).  Calibrated on
// GB300 (CUDA-graph replay, no epilogue): 2048 x 8960 x 1536, 41.1 us in 6
// waves of 24 K blocks; 4096^3, 94.4 us in 6 waves of 64 K blocks.
constexpr double kW4tEfficiency = 0.70;
constexpr double kW4tTileUs = 0.9;

// FP16 x FP16 tiles also compiled with stream-K work division
bool tc_streamk_variant(const TcVariant& v) {
  return (v.n_tile == 256 && v.stages == 6 && v.cta_group == 2) ||
         (v.n_tile == 128 && v.stages == 6 && v.cta_group == 1);
}
// Stream-K ranges are at least this many K blocks long, and a tile with
// fewer tiles than units is cut into at most kSkMaxPieces ranges
constexpr int64_t kSkMinIters = 4;
constexpr int64_t kSkMaxPieces = 4;
// Cost of a split tile per extra piece and accumulator element of the tile
// (microseconds): the writers' partial stores competing with their next
// main loop, and the finisher's exposed read and add before its epilogue.
// Calibrated on GB300 against the data-parallel kernel of every FP16 tile
// (CUDA-graph replay): 256 x 256 pair tiles lost 8-10 us a launch at 2048^3,
// 2560^2 x 4096, 3072^2 x 4096 and 4096^3 and won 30 us at 8192^3; 128 x 128
// tiles won 8 us at 128 and 256 x 4096 x 16384.
constexpr double kSkFixUsPerElem = 1.15e-4;
// and a fixed cost of a launch with split tiles (flag hand-off, the
// finisher's wait): with equal pieces per tile, 128 x 128 tiles measured 1.5
// to 7.6 us above the model on eight shapes where the data-parallel plan
// measured -2.4 to 6.2 us above it (K = 3000 to 32768, 6 to 64 tiles)
constexpr double kSkFixedUs = 3.0;
constexpr TcVariant kTcVariantsI8[] = {{128, 8, 1, 3}};
// FP16 kernel in its exact-INT32 mode (two FP32 chunk accumulators in TMEM,
// running INT32 sums in registers, 32 per 32-column chunk a warp owns: at most
// 96 per thread, so N_tile 128 or 192, or 224 with the last chunk's sums kept
// in a staging box during the tile)
constexpr TcVariant kTcVariantsI8Widened[] = {{128, 6, 1, 0}, {192, 6, 2, 0}, {224, 6, 2, 0}};
constexpr TcVariant kTcVariantsE2M1[] = {{256, 6, 1, 2}, {128, 8, 1, 3}, {64, 8, 1, 4}};
// MXFP4 x MXFP4 on the block-scaled MMA (the tensor-core kernel with packed
// E2M1 stages and scale images; single CTAs)
constexpr TcVariant kTcVariantsMx[] = {{224, 3, 1, 0}, {128, 5, 1, 0}, {224, 5, 2, 0},
                                       {192, 5, 2, 0}};
// E2M1 values per MMA FLOP relative to FP16: the block-scaled 4-bit MMA runs
// at four times the 16-bit rate (the nominal Blackwell ratio)
constexpr double kMxRateRatio = 4.0;
constexpr int kTcBlockM = 128;
constexpr int kTcBlockK = 64;
constexpr int kTcThreads = 384;      // FP16 x FP16 kernel (eight epilogue warps)
constexpr int kConvThreads = 384;    // converting kernel (adds four converter warps)
// Registers per thread: the kernels' own figures (cudaFuncGetAttributes) when
// a device is present to read them from, else these upper bounds of what
// ptxas assigns them.
constexpr int kTcRegsPerThread = 168;
constexpr int kTcBarrierBytes = 512;

struct TcFamily {
  const TcVariant* v;
  int n;
  int threads;
};

TcFamily tc_family(dg_dtype da, dg_dtype db) {
  if (da == DG_F16 && db == DG_F16) return {kTcVariantsF16, kNumTcVariantsF16, kTcThreads};
  if (da == DG_I8 && db == DG_I8) return {kTcVariantsI8, 1, kConvThreads};
  if (da == DG_F16 && db == DG_E2M1) return {kTcVariantsE2M1, 3, kConvThreads};
  if (da == DG_MXF4 && db == DG_MXF4) return {kTcVariantsMx, 4, kTcThreads};
  return {nullptr, 0, 0};
}

// Shared memory of one CTA.  FP16 x FP16: `stages` slots of FP16 tiles
// (128-byte swizzle; a CTA of a pair holds half of the B tile).  Converting
// kernel: `stages` input slots as loaded (FP16 A or raw int8 A; raw int8 /
// packed-E2M1 B) plus `cv_stages` slots of widened FP16 operands.
int tc_ring_bytes(dg_dtype da, dg_dtype db, const TcVariant& v) {
  const int a16 = kTcBlockM * kTcBlockK * 2;
  if (da == DG_MXF4 && db == DG_MXF4)  // 128-byte rows of codes (a CTA of a pair holds half
                                       // of B's), the scale images (the whole B tile's)
                                       // and the row-major scale bytes they are built
                                       // from (16 per row of A and of the B tile)
    return v.stages * (a16 + (v.n_tile / v.cta_group) * kTcBlockK * 2 +
                       1024 * (1 + (v.n_tile + 127) / 128) + 16 * (kTcBlockM + v.n_tile));
  if (da == DG_F16 && db == DG_F16)
    return v.stages * (a16 + (v.n_tile / v.cta_group) * kTcBlockK * 2);
  const int in_a = da == DG_I8 ? kTcBlockM * kTcBlockK : a16;
  const int in_b = db == DG_I8 ? v.n_tile * kTcBlockK : v.n_tile * kTcBlockK / 2;
  const int cv = (da == DG_I8 ? a16 : 0) + v.n_tile * kTcBlockK * 2;
  return v.stages * (in_a + in_b) + v.cv_stages * cv;
}

// Tensor-memory columns: two FP32 accumulators, plus INT32 running sums in the
// converting INT8 kernel (the FP16 kernel's INT32 mode keeps them in registers),
// or two buffers of scale words (8 columns for A, 8 per 128 rows of B) for MXFP4.
int tc_tmem_cols(bool conv_i8, bool mx, int n_tile) {
  if (mx) return 2 * n_tile + 2 * (8 + 8 * ((n_tile + 127) / 128));
  return (conv_i8 ? 3 : 2) * n_tile;
}

constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kGemvRegsPerThread = 64;
constexpr int kGemvMaxM = 8;
constexpr int kGemvResidentWarpsPerSm = 64;
// Split-K counts the GEMV may use: dense at the low end so that a warp's K
// range can match one batch of in-flight loads (1024 K per lane group).
constexpr int kGemvSplits[] = {1,  2,  3,  4,  5,  6,  7,  8,   10,  12,  13,  14,  16,
                               20, 24, 28, 32, 40, 48, 64, 96, 128, 160, 192, 256};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// FP16-output runs of the FP16 x FP16 kernel add the staging boxes of its
// epilogue: two 32 x 32 FP16 boxes for each of the eight epilogue warps.
constexpr int kTcEpiStagingBytes = 8 * 2 * 32 * 32 * 2;

int tc_smem_bytes(dg_dtype da, dg_dtype db, const TcVariant& v, bool staged) {
  return tc_ring_bytes(da, db, v) + (staged ? kTcEpiStagingBytes : 0) + kTcBarrierBytes + 1024;
}

double sm_rate_flops_per_us(const dg_hw_desc& hw) {
  const double tflops = hw.tc_f16_tflops > 0 ? hw.tc_f16_tflops : 1900.0;
  return tflops * 1e6 / std::max(1, hw.sm_count);  // FLOP per microsecond per SM
}

double hbm_bytes_per_us(const dg_hw_desc& hw) {
  const double gbps = hw.hbm_gbps > 0 ? hw.hbm_gbps : 6800.0;
  return gbps * 1e3;  // GB/s -> bytes per microsecond
}

// Fraction of the tensor rate a tile shape sustains per busy SM, calibrated on
// GB300 at 4096^3 (measured time x wave efficiency): wider tiles and CTA pairs
// move fewer operand bytes through L2 and shared memory per FLOP.
double tc_tile_efficiency(int n_tile, int cta_group, bool mx = false) {
  // block-scaled MXFP4 tiles, calibrated at 8192^3: single CTAs 128 x 224
  // ran 1.17x as fast as 128 x 128 per FLOP (199 against 233 us), CTA pairs
  // 256 x 224 and 256 x 192 took 184 and 191 us against 210 for 128 x 224
  if (mx && cta_group == 2) return n_tile >= 224 ? 0.98 : 0.945;
  if (mx) return n_tile >= 224 ? 0.86 : 0.73;
  if (cta_group == 2) return n_tile >= 224 ? 0.86 : (n_tile >= 192 ? 0.80 : 0.63);
  switch (n_tile) {
    case 256: return 0.72;
    case 128: return 0.57;
    default: return 0.40;
  }
}

// Tensor-core candidates.  widened == false: the kernel that reads the
// operands as stored (FP16 x FP16, or the converting kernel that widens
// int8 / E2M1 tiles in shared memory).  widened == true (int8 / E2M1 only):
// a streaming pre-pass widens the narrow operands to FP16 in a workspace and
// the FP16 kernel runs on the copies (INT8 with its exact INT32 output mode).
void add_tc_candidates(int64_t M, int64_t N, int64_t K, dg_dtype da, dg_dtype db, bool widened,
                       const dg_hw_desc& hw, double target, std::vector<dg_tile_plan>* out,
                       std::string* why) {
  const bool narrow = !(da == DG_F16 && db == DG_F16);
  if (widened && !narrow) return;
  if ((da == DG_MXF4) != (db == DG_MXF4)) return;
  // MXFP4 runs natively on the block-scaled MMA, or widened to BF16 on the
  // 16-bit tiles; the native kernel reads whole bytes of codes, so an odd K
  // (half a byte past the end of each row) runs widened
  const bool mx_native = da == DG_MXF4 && !widened;
  if (mx_native && K % 2 != 0) {
    if (why) *why += "block-scaled MXFP4: odd K; ";
    return;
  }
  constexpr int kNumI8Widened = sizeof(kTcVariantsI8Widened) / sizeof(TcVariant);
  TcFamily fam = widened ? (da == DG_I8 ? TcFamily{kTcVariantsI8Widened, kNumI8Widened, kTcThreads}
                                        : TcFamily{kTcVariantsF16, kNumTcVariantsF16, kTcThreads})
                         : tc_family(da, db);
  if (!fam.v) {
    if (why) *why += "tensor-core kernel: dtype pair not compiled; ";
    return;
  }
  if (hw.cc_major < 10 || hw.tmem_cols <= 0) {
    if (why) *why += "tensor-core kernel: needs tcgen05 / tensor memory; ";
    return;
  }
  // bytes per element read from HBM for A and B (MXFP4: half a byte of code
  // and a 32nd of a scale byte)
  const double mx_elem = 0.5 + 1.0 / 32.0;
  const double elem_a = da == DG_I8 ? 1.0 : (da == DG_MXF4 ? mx_elem : 2.0);
  const double elem_b =
      db == DG_I8 ? 1.0 : (db == DG_E2M1 ? 0.5 : (db == DG_MXF4 ? mx_elem : 2.0));
  const double elem_d = da == DG_I8 ? 4.0 : 2.0;
  // the pre-pass reads the narrow operands and writes 16-bit copies (an FP16
  // A is used as it is)
  const double pre_bytes =
      widened ? (da == DG_F16 ? 0.0 : (elem_a + 2.0) * M * static_cast<double>(K)) +
                    (elem_b + 2.0) * N * static_cast<double>(K)
              : 0.0;
  const double t_pre = widened ? pre_bytes / hbm_bytes_per_us(hw) + (da == DG_I8 ? 4.0 : 2.0) : 0.0;
  // shared memory / tensor memory are those of the kernel that runs
  const dg_dtype ka = widened ? DG_F16 : da, kb = widened ? DG_F16 : db;
  for (int vi = 0; vi < fam.n; ++vi) {
    const TcVariant& v = fam.v[vi];
    const std::string name = std::string(widened ? "widened " : "") + "N_tile " +
                             std::to_string(v.n_tile) + (v.cta_group == 2 ? " (CTA pair)" : "");
    if (v.cta_group == 2 && M <= kTcBlockM) {
      if (why) *why += name + ": M fits one CTA; ";
      continue;
    }
    // the FP16 x FP16 kernel stages its output (FP16, or INT32 for widened
    // INT8), and so does the MXFP4 kernel
    const bool staged = (ka == DG_F16 && kb == DG_F16) || mx_native;
    const int smem = tc_smem_bytes(ka, kb, v, staged);
    if (smem > hw.smem_per_block_optin) {
      if (why) *why += name + ": shared memory; ";
      continue;
    }
    if (tc_tmem_cols(da == DG_I8 && !widened, mx_native, v.n_tile) > hw.tmem_cols) {
      if (why) *why += name + ": tensor memory; ";
      continue;
    }
    const int measured = mx_native ? mx_kernel_regs(v.n_tile, v.stages, v.cta_group)
                         : (ka == DG_F16 && kb == DG_F16)
                             ? tc_kernel_regs(v.n_tile, v.stages, v.cta_group,
                                              widened && da == DG_I8)
                             : conv_kernel_regs(ka, kb, v.n_tile, v.stages);
    const int regs = measured > 0 ? measured : kTcRegsPerThread;
    if (regs > hw.regs_per_thread_max || regs * fam.threads > hw.regs_per_sm) {
      if (why) *why += name + ": registers; ";
      continue;
    }
    // A pair works on 256-row tiles with half the SMs as scheduling units.
    const int tile_m = kTcBlockM * v.cta_group;
    const int64_t units = std::max(1, hw.sm_count / v.cta_group);
    const int64_t tiles = ceil_div(M, tile_m) * ceil_div(N, v.n_tile);
    const int64_t waves = ceil_div(tiles, units);
    const double occ = static_cast<double>(tiles) / static_cast<double>(waves * units);
    const int64_t k_step = mx_native ? 256 : kTcBlockK;  // K per pipeline stage
    const int64_t k_pad = ceil_div(K, k_step) * k_step;
    // FLOPs of one tile per SM of its unit
    const double tile_flops = 2.0 * kTcBlockM * v.n_tile * static_cast<double>(k_pad);
    const double t_tile =
        tile_flops / (sm_rate_flops_per_us(hw) * tc_tile_efficiency(v.n_tile, v.cta_group));
    const double t_epi = (128.0 * v.n_tile * 4.0) / (hbm_bytes_per_us(hw) / hw.sm_count);
    if (!widened && !narrow && tc_streamk_variant(v) && tiles < units) {
      // The same tile with stream-K division: the K blocks in one even range
      // per unit; a split tile costs its finisher the read of the other
      // ranges' partials.  Proposed only when the tiles do not fill one wave:
      // with more tiles than units the ranges start at scattered K offsets,
      // units that share an operand panel no longer read it in step, and the
      // panels are read again from DRAM (FP16 8192^3: 1.69 GB a launch
      // against 1.09 GB for the data-parallel plan, measured on GB300),
      // which the power cap turns into lost clock: 1501 against 1492 TFLOP/s
      // under a sustained load.  Forced plans may still divide whole waves
      // plus ranges.
      const int64_t kbn = k_pad / k_step;
      const SkSplit sp = stream_k_split(tiles, kbn, units);
      const int sk_regs = tc_streamk_kernel_regs(v.n_tile, v.stages, v.cta_group);
      const int regs_sk = sk_regs > 0 ? sk_regs : kTcRegsPerThread;
      if (sp.sk_tiles > 0 && regs_sk <= hw.regs_per_thread_max &&
          regs_sk * fam.threads <= hw.regs_per_sm) {
        const int64_t range = ceil_div(sp.sk_iters, sp.sk_units);
        const double unit_iters = static_cast<double>(sp.dp_tiles / units * kbn + range);
        const double occ_sk = static_cast<double>(tiles * kbn) / (units * unit_iters);
        if (occ_sk >= target) {
          const double t_math = unit_iters / kbn * t_tile;
          const double t_fix =
              sp.max_pieces > 1
                  ? kSkFixedUs + (sp.max_pieces - 1) * static_cast<double>(tile_m) * v.n_tile *
                                     kSkFixUsPerElem
                  : 0.0;
          const double bytes = 2.0 * (M * K + N * K) + 4.0 * M * N;
          dg_tile_plan q{};
          q.kernel = DG_KERNEL_TC_STREAMK;
          q.m_tile = tile_m;
          q.n_tile = v.n_tile;
          q.k_tile = static_cast<int>(k_step);
          q.split_k = sp.max_pieces;
          q.stages = v.stages;
          q.cta_group = v.cta_group;
          q.swap_ab = 0;
          q.smem_bytes = tc_smem_bytes(ka, kb, v, true);
          q.threads = fam.threads;
          q.regs_per_thread = regs_sk;
          q.grid = static_cast<int>(units * v.cta_group);  // the units the work is divided over
          q.occupancy = occ_sk;
          q.est_us = std::max(t_math, bytes / hbm_bytes_per_us(hw)) + t_epi + 2.0 + t_fix;
          q.est_tflops = 2.0 * M * N * K / (q.est_us * 1e6);
          out->push_back(q);
        }
      }
    }
    if (occ < target) {
      if (why) *why += name + ": occupancy; ";
      continue;
    }
    // The converting kernel spends shared-memory bandwidth and issue slots
    // widening tiles (calibrated on GB300: INT8 4096^3; W4A16 at M = 64 and
    // 128 x 8960 x 1536, 11.7 and 11.9 us).
    const double conv_eff = mx_native ? kMxRateRatio
                            : (narrow && !widened) ? (da == DG_I8 ? 0.36 : 0.44)
                                                   : 1.0;
    const double t_math =
        waves * tile_flops /
        (sm_rate_flops_per_us(hw) * tc_tile_efficiency(v.n_tile, v.cta_group, mx_native) *
         conv_eff);
    const double bytes = elem_a * M * K + elem_b * N * K + 2.0 * M * N * elem_d;
    const double t_mem = bytes / hbm_bytes_per_us(hw);
    dg_tile_plan p{};
    p.kernel = widened ? DG_KERNEL_TC_WIDENED : DG_KERNEL_TC;
    p.m_tile = tile_m;
    p.n_tile = v.n_tile;
    p.k_tile = static_cast<int>(k_step);
    p.split_k = 1;
    p.stages = v.stages;
    p.cta_group = v.cta_group;
    p.swap_ab = 0;
    p.smem_bytes = smem;
    p.threads = fam.threads;
    p.regs_per_thread = regs;
    p.grid = static_cast<int>(std::min<int64_t>(tiles, units) * v.cta_group);
    p.occupancy = occ;
    p.est_us = std::max(t_math, t_mem) + t_epi + 2.0 + t_pre;
    p.est_tflops = 2.0 * M * N * K / (p.est_us * 1e6);
    out->push_back(p);
  }
}

int w4t_smem_bytes(const TcVariant& v) {
  return v.stages * (v.n_tile * kTcBlockK * 2 + kTcBlockM * kTcBlockK / 2) +
         8 * 2 * 32 * 32 * 2 + 1024 + 512;
}

// FP16 x E2M1 with the weights widened in tensor memory: D^T tiles of 128
// weight rows x n_tile activation rows, one CTA per SM.
void add_w4t_candidates(int64_t M, int64_t N, int64_t K, dg_dtype da, dg_dtype db,
                        const dg_hw_desc& hw, double target, std::vector<dg_tile_plan>* out,
                        std::string* why) {
  if (!(da == DG_F16 && db == DG_E2M1) || hw.cc_major < 10 || hw.tmem_cols <= 0) return;
  for (const TcVariant& v : kW4tVariants) {
    const std::string name = "tensor-memory widening N_tile " + std::to_string(v.n_tile);
    const int smem = w4t_smem_bytes(v);
    if (smem > hw.smem_per_block_optin) {
      if (why) *why += name + ": shared memory; ";
      continue;
    }
    if (2 * v.n_tile + 2 * 32 > hw.tmem_cols) {  // two accumulators and two A slots
      if (why) *why += name + ": tensor memory; ";
      continue;
    }
    const int measured = w4t_kernel_regs(v.n_tile, v.stages);
    const int regs = measured > 0 ? measured : 144;
    if (regs > hw.regs_per_thread_max || regs * kW4tThreads > hw.regs_per_sm) {
      if (why) *why += name + ": registers; ";
      continue;
    }
    const int64_t units = std::max(1, hw.sm_count);
    const int64_t tiles = ceil_div(N, kTcBlockM) * ceil_div(M, v.n_tile);
    const int64_t waves = ceil_div(tiles, units);
    const double occ = static_cast<double>(tiles) / static_cast<double>(waves * units);
    if (occ < target) {
      if (why) *why += name + ": occupancy; ";
      continue;
    }
    const int64_t kbn = ceil_div(K, kTcBlockK);
    const double t_stage = 2.0 * kTcBlockM * v.n_tile * kTcBlockK /
                           (sm_rate_flops_per_us(hw) * kW4tEfficiency);
    const double t_math = waves * (kW4tTileUs + kbn * t_stage);
    const double bytes = 2.0 * M * K + 0.5 * N * K + 2.0 * M * N;
    const double t_mem = bytes / hbm_bytes_per_us(hw);
    const double t_epi = (128.0 * v.n_tile * 4.0) / (hbm_bytes_per_us(hw) / hw.sm_count);
    dg_tile_plan p{};
    p.kernel = DG_KERNEL_TC;
    p.m_tile = kTcBlockM;
    p.n_tile = v.n_tile;
    p.k_tile = kTcBlockK;
    p.split_k = 1;
    p.stages = v.stages;
    p.cta_group = 1;
    p.swap_ab = 1;
    p.smem_bytes = smem;
    p.threads = kW4tThreads;
    p.regs_per_thread = regs;
    p.grid = static_cast<int>(std::min<int64_t>(tiles, units));
    p.occupancy = occ;
    p.est_us = std::max(t_math, t_mem) + t_epi + 2.0;
    p.est_tflops = 2.0 * M * N * K / (p.est_us * 1e6);
    out->push_back(p);
  }
}

void add_gemv_candidates(int64_t M, int64_t N, int64_t K, dg_dtype da, dg_dtype db,
                         const dg_hw_desc& hw, double target, std::vector<dg_tile_plan>* out,
                         std::string* why) {
  if (!(da == DG_F16 && db == DG_F16)) {
    if (why) *why += "GEMV: dtype pair not compiled; ";
    return;
  }
  if (M > kGemvMaxM) {
    if (why) *why += "GEMV: M > 8; ";
    return;
  }
  const int64_t resident = static_cast<int64_t>(hw.sm_count) * kGemvResidentWarpsPerSm;
  for (int split : kGemvSplits) {
    // splits of 2 .. 8 run the cluster-reduction variant, the others the
    // global-memory one: each its own register figure
    const int measured = gemv_kernel_regs(M, split);
    const int regs = measured > 0 ? measured : kGemvRegsPerThread;
    if (regs * kGemvThreads > hw.regs_per_sm) {
      if (why) *why += "GEMV split " + std::to_string(split) + ": registers; ";
      continue;
    }
    int64_t chunk = 0;
    const double t = gemv_estimate_us(M, N, K, split, hw, &chunk);
    if (t < 0) continue;  // the last split would be empty
    const int64_t units = N * split;  // warps
    const int64_t waves = ceil_div(units, resident);
    const double occ = static_cast<double>(units) / static_cast<double>(waves * resident);
    if (occ < target) {
      if (why) *why += "GEMV split " + std::to_string(split) + ": occupancy; ";
      continue;
    }
    dg_tile_plan p{};
    p.kernel = DG_KERNEL_GEMV;
    p.m_tile = static_cast<int>(M);
    p.n_tile = kGemvWarps;
    p.k_tile = static_cast<int>(chunk);
    p.split_k = split;
    p.stages = 1;
    p.cta_group = 1;
    p.swap_ab = 0;
    p.smem_bytes = 0;
    p.threads = kGemvThreads;
    p.regs_per_thread = regs;
    p.grid = static_cast<int>(ceil_div(N, kGemvWarps) * split);
    p.occupancy = occ;
    p.est_us = t;
    p.est_tflops = 2.0 * M * N * K / (t * 1e6);
    out->push_back(p);
  }
}

// Warp-MMA GEMV (FP16 x FP16, 2 <= M <= 16): CTAs of 8 warps, a warp owns 8
// output columns and streams their 8 rows of B in batches of 8 x 32 K.
constexpr int kGemvMmaMinM = 2;
constexpr int kGemvMmaMaxM = 16;
constexpr int kGemvMmaCols = 64;
constexpr int kGemvMmaThreads = 256;
constexpr int kGemvMmaRegsPerThread = 80;  // upper bound of what ptxas assigns the kernel

int gemv_mma_regs(int64_t M) {
  const int measured = gemv_mma_kernel_regs(M);
  return measured > 0 ? measured : kGemvMmaRegsPerThread;
}

void add_gemv_mma_candidates(int64_t M, int64_t N, int64_t K, dg_dtype da, dg_dtype db,
                             const dg_hw_desc& hw, double target, std::vector<dg_tile_plan>* out,
                             std::string* why) {
  if (!(da == DG_F16 && db == DG_F16)) return;
  if (M < kGemvMmaMinM || M > kGemvMmaMaxM) {
    if (why) *why += "warp-MMA GEMV: M outside [2, 16]; ";
    return;
  }
  const int regs = gemv_mma_regs(M);
  const int ctas = hw.regs_per_sm / (regs * kGemvMmaThreads);
  if (ctas < 1) {
    if (why) *why += "warp-MMA GEMV: registers; ";
    return;
  }
  const int64_t resident = static_cast<int64_t>(hw.sm_count) * ctas * (kGemvMmaThreads / 32);
  for (int split : kGemvSplits) {
    int64_t chunk = 0;
    const double t = gemv_mma_estimate_us(M, N, K, split, hw, &chunk);
    if (t < 0) continue;
    const int64_t units = ceil_div(N, 8) * split;  // warps
    const int64_t waves = ceil_div(units, resident);
    const double occ = static_cast<double>(units) / static_cast<double>(waves * resident);
    if (occ < target) {
      if (why) *why += "warp-MMA GEMV split " + std::to_string(split) + ": occupancy; ";
      continue;
    }
    dg_tile_plan p{};
    p.kernel = DG_KERNEL_GEMV_MMA;
    p.m_tile = kGemvMmaMaxM;
    p.n_tile = kGemvMmaCols;
    p.k_tile = static_cast<int>(chunk);
    p.split_k = split;
    p.stages = 1;
    p.cta_group = 1;
    p.smem_bytes = 0;
    p.threads = kGemvMmaThreads;
    p.regs_per_thread = regs;
    p.grid = static_cast<int>(ceil_div(N, kGemvMmaCols) * split);
    p.occupancy = occ;
    p.est_us = t;
    p.est_tflops = 2.0 * M * N * K / (t * 1e6);
    out->push_back(p);
  }
}

// Skinny W4A16 kernel: FP16 A with M <= 16 rows x packed E2M1 B, one block
// of 512 threads per 64 columns, K in 2048-code chunks split between two warp
// halves; the weights stream from HBM once.
constexpr int kSkinnyMaxM = 16;
constexpr int kSkinnyRegsPerThread = 80;

void add_skinny_candidates(int64_t M, int64_t N, int64_t K, dg_dtype da, dg_dtype db,
                           const dg_hw_desc& hw, double target, std::vector<dg_tile_plan>* out,
                           std::string* why) {
  if (!(da == DG_F16 && db == DG_E2M1)) return;
  if (M > kSkinnyMaxM) {
    if (why) *why += "skinny: M > 16; ";
    return;
  }
  if (hw.cc_major < 8) {
    if (why) *why += "skinny: needs m16n8k16 FP16 MMA; ";
    return;
  }
  const int smem = skinny_smem_bytes();
  if (smem > hw.smem_per_block_optin) {
    if (why) *why += "skinny: shared memory; ";
    return;
  }
  const int threads = skinny_threads();
  const int measured = skinny_kernel_regs();
  const int regs = measured > 0 ? measured : kSkinnyRegsPerThread;
  if (regs * threads > hw.regs_per_sm) {
    if (why) *why += "skinny: registers; ";
    return;
  }
  const int64_t blocks = ceil_div(N, skinny_cols_per_block());
  const int64_t per_sm = std::max<int64_t>(
      1, std::min<int64_t>(hw.smem_per_sm / smem, hw.max_threads_per_sm / threads));
  const int64_t slots = per_sm * hw.sm_count;
  const int64_t waves = ceil_div(blocks, slots);
  const double occ = static_cast<double>(blocks) / static_cast<double>(waves * slots);
  if (occ < target) {
    if (why) *why += "skinny: occupancy; ";
    return;
  }
  // Streaming time of the weights over the SMs that hold a block, plus a
  // fixed latency (launch, activation load, one round trip per chunk).
  const double busy = std::min(1.0, static_cast<double>(blocks) / hw.sm_count);
  const double bytes = 0.5 * N * static_cast<double>(K) + 2.0 * M * K + 2.0 * M * N;
  const int64_t chunks = ceil_div(K, skinny_k_chunk());
  const double t = 2.0 + 1.0 * static_cast<double>(chunks) +
                   bytes / (hbm_bytes_per_us(hw) * 0.8 * busy);
  dg_tile_plan p{};
  p.kernel = DG_KERNEL_SKINNY;
  p.m_tile = kSkinnyMaxM;
  p.n_tile = skinny_cols_per_block();
  p.k_tile = skinny_k_chunk();
  p.split_k = 2;
  p.stages = 1;
  p.cta_group = 1;
  p.swap_ab = 0;
  p.smem_bytes = smem;
  p.threads = threads;
  p.regs_per_thread = regs;
  p.grid = static_cast<int>(blocks);
  p.occupancy = occ;
  p.est_us = t;
  p.est_tflops = 2.0 * M * N * K / (t * 1e6);
  out->push_back(p);
}

// Warp-level-MMA tile family for GPUs without tensor memory (planning only).
void add_warp_mma_candidates(int64_t M, int64_t N, int64_t K, dg_dtype da, const dg_hw_desc& hw,
                             double target, std::vector<dg_tile_plan>* out, std::string* why) {
  const int elem = (da == DG_I8) ? 1 : 2;
  const int max_warps = std::max(1, hw.max_threads_per_sm / 32);
  const int sizes_mn[] = {16, 32, 48, 64, 80, 96, 112, 128};
  const int sizes_k[] = {16, 32, 48, 64};
  for (int mt : sizes_mn) {
    for (int nt : sizes_mn) {
      for (int kt : sizes_k) {
        const int stages = 2;
        // One warp per 32 x 32 block of outputs (at least one warp).
        const int warps = std::max(1, (mt * nt) / 1024);
        const int threads = warps * 32;
        const int smem = stages * (mt + nt) * kt * elem;
        const int acc_regs = (mt * nt) / threads;  // FP32 accumulators per thread
        const int regs = 32 + acc_regs + (mt + nt) * kt * elem / (4 * threads) + 16;
        if (smem > hw.smem_per_block_optin || regs > hw.regs_per_thread_max) continue;
        int ctas = std::min(hw.smem_per_sm / std::max(1, smem), hw.max_threads_per_sm / threads);
        ctas = std::min(ctas, hw.regs_per_sm / (regs * threads));
        ctas = std::min(ctas, 32);
        if (ctas < 1) continue;
        const double occ = std::min(1.0, static_cast<double>(ctas * warps) / max_warps);
        if (occ < target) continue;
        const int64_t tiles = ceil_div(M, mt) * ceil_div(N, nt);
        const int64_t slots = static_cast<int64_t>(hw.sm_count) * ctas;
        const int64_t waves = ceil_div(tiles, slots);
        // Operand re-reads from L2 per tile grow as tiles shrink.
        const double l2_bytes = static_cast<double>(tiles) * (mt + nt) * K * elem;
        const double rate = sm_rate_flops_per_us(hw) * hw.sm_count;
        const double t_math = 2.0 * M * N * K / rate *
                              static_cast<double>(waves * slots) / static_cast<double>(tiles);
        const double t_l2 = l2_bytes / (4.0 * hbm_bytes_per_us(hw));
        dg_tile_plan p{};
        p.kernel = -1;  // no kernel in this library
        p.m_tile = mt;
        p.n_tile = nt;
        p.k_tile = kt;
        p.split_k = 1;
        p.stages = stages;
        p.cta_group = 1;
        p.smem_bytes = smem;
        p.threads = threads;
        p.regs_per_thread = regs;
        p.grid = static_cast<int>(std::min<int64_t>(tiles, slots));
        p.occupancy = occ;
        p.est_us = std::max(t_math, t_l2) + 2.0;
        p.est_tflops = 2.0 * M * N * K / (p.est_us * 1e6);
        out->push_back(p);
      }
    }
  }
  if (out->empty() && why) *why += "warp-MMA family: no tile meets every constraint; ";
}

}  // namespace

// Cost model of the split-K GEMV for one split count.  K per split is a
// multiple of 256 (one warp-wide step of 8 elements per lane).  Each warp
// keeps about 2 KB in flight (~2 GB/s); HBM caps the total.  Returns a
// negative value when the last split would be empty.  Allocates nothing.
double gemv_estimate_us(int64_t M, int64_t N, int64_t K, int split, const dg_hw_desc& hw,
                        int64_t* chunk_out, int64_t batch) {
  const int64_t kk = K > 0 ? K : 1;
  const int64_t chunk = ceil_div(ceil_div(kk, split), 256) * 256;
  if (split > 1 && chunk * (split - 1) >= kk) return -1.0;
  if (chunk_out) *chunk_out = chunk;
  const int64_t resident = static_cast<int64_t>(hw.sm_count) * kGemvResidentWarpsPerSm;
  const int64_t units = N * split * batch;
  const double active = static_cast<double>(std::min(units, resident));
  const double bw = std::min(hbm_bytes_per_us(hw), active * 2.0e3);
  // Splits of 2 .. 8 reduce in a thread-block cluster through distributed
  // shared memory (no partial sums in global memory, one cluster barrier);
  // more splits write FP32 partials that the last CTA of a row group reads
  // back.
  const bool cluster = split >= 2 && split <= 8;
  const double partial_bytes = (split > 1 && !cluster) ? 8.0 * split * M * N : 0.0;
  const double bytes = batch * (2.0 * (N * K + M * K) + partial_bytes + 4.0 * M * N);
  // A warp streams its K range in batches of 256-element steps (4 at a time,
  // 8 in the cluster variant), one memory round trip (~0.8 us) each; small
  // problems are bound by that latency.
  const double batches = static_cast<double>(ceil_div(chunk, cluster ? 2048 : 1024));
  // Each further row of A costs the FMA loop about 0.65 of the one-row time
  // (measured on GB300 at M = 2..8: 1.7x, 3.0x, 5.8x at M = 2, 4, 8).
  const double rows = 1.0 + 0.65 * static_cast<double>(M - 1);
  const double reduce = split == 1 ? 0.0 : (cluster ? 0.3 : 1.0);
  return std::max(bytes / bw, 0.8 * batches) * rows + reduce + 2.0;
}

double gemv_mma_estimate_us(int64_t M, int64_t N, int64_t K, int split, const dg_hw_desc& hw,
                            int64_t* chunk_out, int64_t batch) {
  const int64_t kk = K > 0 ? K : 1;
  const int64_t chunk = ceil_div(ceil_div(kk, split), 256) * 256;
  if (split > 1 && chunk * (split - 1) >= kk) return -1.0;
  if (chunk_out) *chunk_out = chunk;
  const int ctas = std::max(1, hw.regs_per_sm / (gemv_mma_regs(M) * kGemvMmaThreads));
  const int64_t resident = static_cast<int64_t>(hw.sm_count) * ctas * (kGemvMmaThreads / 32);
  const int64_t units = ceil_div(N, 8) * split * batch;  // warps
  // A warp keeps 8 rows x 8 steps x 64 bytes = 4 KB in flight; measured on
  // GB300 it moves about 2 KB per us.  Warps beyond one resident wave run in
  // later waves.
  const int64_t waves = ceil_div(units, resident);
  const double per_wave = static_cast<double>(std::min(units, resident));
  const double bw = std::min(hbm_bytes_per_us(hw), per_wave * 2.0e3);
  const double bytes = batch * (2.0 * (N * K + M * K) + (split > 1 ? 8.0 * split * M * N : 0.0) +
                                4.0 * M * N);
  const double t_mem = waves * (bytes * per_wave / static_cast<double>(units)) / bw;
  const double batches = static_cast<double>(ceil_div(chunk, 256));
  // Fixed costs measured on GB300: about 6 us of launch, ramp and tail; the
  // 16-row variant (M > 8) streams about 1.2x slower than the 8-row one.
  const double rows = M > 8 ? 1.2 : 1.0;
  return std::max(t_mem, 0.8 * batches * waves) * rows + (split > 1 ? 1.0 : 0.0) + 6.0;
}

int gemv_mma_best_split(int64_t M, int64_t N, int64_t K, const dg_hw_desc& hw,
                        int64_t* chunk_out, int64_t batch) {
  int best = 1;
  double best_t = -1.0;
  for (int split : kGemvSplits) {
    int64_t chunk = 0;
    const double t = gemv_mma_estimate_us(M, N, K, split, hw, &chunk, batch);
    if (t < 0) continue;
    if (best_t < 0 || t < best_t) {
      best_t = t;
      best = split;
      if (chunk_out) *chunk_out = chunk;
    }
  }
  return best;
}

int gemv_best_split(int64_t M, int64_t N, int64_t K, const dg_hw_desc& hw, int64_t* chunk_out,
                    int64_t batch) {
  int best = 1;
  double best_t = -1.0;
  for (int split : kGemvSplits) {
    int64_t chunk = 0;
    const double t = gemv_estimate_us(M, N, K, split, hw, &chunk, batch);
    if (t < 0) continue;
    if (best_t < 0 || t < best_t) {
      best_t = t;
      best = split;
      if (chunk_out) *chunk_out = chunk;
    }
  }
  return best;
}

SkSplit stream_k_split(int64_t tiles, int64_t kblocks, int64_t units) {
  SkSplit s{tiles, 0, 0, 0, 1};
  if (tiles < 1 || kblocks < 2 || units < 2 || tiles % units == 0) return s;
  int64_t u;
  if (tiles < units) {
    // Fewer tiles than units: every tile cut into p equal K ranges (p units
    // per tile, at most kSkMaxPieces, ranges of at least kSkMinIters K
    // blocks).  Ranges then never straddle two tiles, and the units holding
    // the same piece of tiles that share an operand panel read the same K
    // slices of it at the same time, so each byte crosses DRAM once (with
    // ranges at scattered offsets the panels were read again: 256 x 4096 x
    // 16384 in 128 x 128 tiles took 53 us with 152 ranges, 41 us with two
    // pieces per tile).
    const int64_t p = std::min<int64_t>(std::min<int64_t>(units / tiles, kSkMaxPieces),
                                        kblocks / kSkMinIters);
    if (p < 2) return s;
    s.sk_tiles = tiles;
    s.dp_tiles = 0;
    u = tiles * p;
  } else {
    // the last, ragged wave and the whole wave before it, so that every
    // range is at least one tile long; ranges of at least half a tile and
    // at least kSkMinIters K blocks
    s.sk_tiles = tiles % units + units;
    s.dp_tiles = tiles - s.sk_tiles;
    u = std::min<int64_t>(units, 2 * s.sk_tiles);
    u = std::min<int64_t>(u, std::max<int64_t>(1, s.sk_tiles * kblocks / kSkMinIters));
  }
  s.sk_iters = s.sk_tiles * kblocks;
  s.sk_units = static_cast<int>(u);
  auto unit_of = [&](int64_t i) { return ((i + 1) * u - 1) / s.sk_iters; };
  for (int64_t ts = 0; ts < s.sk_tiles; ++ts) {
    const int64_t pieces = unit_of(ts * kblocks + kblocks - 1) - unit_of(ts * kblocks) + 1;
    s.max_pieces = std::max<int>(s.max_pieces, static_cast<int>(pieces));
  }
  return s;
}

dg_status plan_tiles(int64_t M, int64_t N, int64_t K, dg_dtype dtype_a, dg_dtype dtype_b,
                     dg_epilogue epilogue, const dg_hw_desc& hw, double target_occupancy,
                     dg_tile_plan* out, int max_out, int* n_out, std::string* why) {
  (void)epilogue;
  if (n_out) *n_out = 0;
  std::vector<dg_tile_plan> cands;
  if (hw.tmem_cols > 0) {
    add_tc_candidates(M, N, K, dtype_a, dtype_b, false, hw, target_occupancy, &cands, why);
    add_tc_candidates(M, N, K, dtype_a, dtype_b, true, hw, target_occupancy, &cands, why);
    add_w4t_candidates(M, N, K, dtype_a, dtype_b, hw, target_occupancy, &cands, why);
    add_gemv_candidates(M, N, K, dtype_a, dtype_b, hw, target_occupancy, &cands, why);
    add_gemv_mma_candidates(M, N, K, dtype_a, dtype_b, hw, target_occupancy, &cands, why);
    add_skinny_candidates(M, N, K, dtype_a, dtype_b, hw, target_occupancy, &cands, why);
  } else {
    add_warp_mma_candidates(M, N, K, dtype_a, hw, target_occupancy, &cands, why);
  }
  if (cands.empty()) return DG_ERR_NO_VALID_CANDIDATE;
  std::stable_sort(cands.begin(), cands.end(), [](const dg_tile_plan& a, const dg_tile_plan& b) {
    return a.est_us < b.est_us;
  });
  const int n = std::min<int>(static_cast<int>(cands.size()), std::max(0, max_out));
  for (int i = 0; i < n; ++i) out[i] = cands[i];
  if (n_out) *n_out = (max_out <= 0) ? static_cast<int>(cands.size()) : n;
  return DG_OK;
}

bool plan_is_runnable(const dg_tile_plan& plan, int64_t M, int64_t N, int64_t K,
                      dg_dtype dtype_a, dg_dtype dtype_b, std::string* why) {
  (void)N;
  if (plan.kernel == DG_KERNEL_TC && plan.swap_ab == 1) {
    if (!(dtype_a == DG_F16 && dtype_b == DG_E2M1)) {
      if (why) *why = "tensor-memory widening plans (swap_ab) are for F16 x E2M1";
      return false;
    }
    if (plan.cta_group != 1 || plan.m_tile != kTcBlockM || plan.k_tile != kTcBlockK ||
        plan.split_k != 1) {
      if (why) *why = "tensor-memory widening plan shape not compiled";
      return false;
    }
    for (const TcVariant& v : kW4tVariants)
      if (v.n_tile == plan.n_tile && v.stages == plan.stages) return true;
    if (why) *why = "tensor-memory widening N_tile/stages pair not compiled";
    return false;
  }
  if (plan.kernel == DG_KERNEL_TC) {
    const TcFamily fam = tc_family(dtype_a, dtype_b);
    if (!fam.v) {
      if (why) *why = "tensor-core plan for a dtype pair it does not take";
      return false;
    }
    const bool mx = dtype_a == DG_MXF4;
    if ((plan.cta_group != 1 && plan.cta_group != 2) ||
        plan.m_tile != kTcBlockM * plan.cta_group || plan.k_tile != (mx ? 256 : kTcBlockK) ||
        plan.split_k != 1 || plan.swap_ab != 0) {
      if (why) *why = "tensor-core plan shape not compiled";
      return false;
    }
    if (mx && K % 2 != 0) {
      if (why) *why = "block-scaled MXFP4 plan with an odd K";
      return false;
    }
    for (int vi = 0; vi < fam.n; ++vi)
      if (fam.v[vi].n_tile == plan.n_tile && fam.v[vi].stages == plan.stages &&
          fam.v[vi].cta_group == plan.cta_group)
        return true;
    if (why) *why = "tensor-core N_tile/stages pair not compiled";
    return false;
  }
  if (plan.kernel == DG_KERNEL_TC_STREAMK) {
    if (!(dtype_a == DG_F16 && dtype_b == DG_F16)) {
      if (why) *why = "stream-K plans are for F16 x F16";
      return false;
    }
    if ((plan.cta_group != 1 && plan.cta_group != 2) ||
        plan.m_tile != kTcBlockM * plan.cta_group || plan.k_tile != kTcBlockK ||
        plan.split_k < 1 || plan.swap_ab != 0) {
      if (why) *why = "stream-K plan shape not compiled";
      return false;
    }
    if (!tc_streamk_variant(TcVariant{plan.n_tile, plan.stages, plan.cta_group, 0})) {
      if (why) *why = "stream-K N_tile/stages pair not compiled";
      return false;
    }
    return true;
  }
  if (plan.kernel == DG_KERNEL_TC_WIDENED) {
    const bool i8 = dtype_a == DG_I8 && dtype_b == DG_I8;
    const bool e2m1 = dtype_a == DG_F16 && dtype_b == DG_E2M1;
    const bool mxf4 = dtype_a == DG_MXF4 && dtype_b == DG_MXF4;
    if (!i8 && !e2m1 && !mxf4) {
      if (why) *why = "widened plans are for INT8 x INT8, FP16 x E2M1 and MXF4 x MXF4";
      return false;
    }
    if ((plan.cta_group != 1 && plan.cta_group != 2) ||
        plan.m_tile != kTcBlockM * plan.cta_group || plan.k_tile != kTcBlockK ||
        plan.split_k != 1 || plan.swap_ab != 0) {
      if (why) *why = "widened plan shape not compiled";
      return false;
    }
    const TcVariant* vs = i8 ? kTcVariantsI8Widened : kTcVariantsF16;
    const int n = i8 ? static_cast<int>(sizeof(kTcVariantsI8Widened) / sizeof(TcVariant))
                     : kNumTcVariantsF16;
    for (int vi = 0; vi < n; ++vi)
      if (vs[vi].n_tile == plan.n_tile && vs[vi].stages == plan.stages &&
          vs[vi].cta_group == plan.cta_group)
        return true;
    if (why) *why = "widened N_tile/stages pair not compiled";
    return false;
  }
  if (plan.kernel == DG_KERNEL_SKINNY) {
    if (!(dtype_a == DG_F16 && dtype_b == DG_E2M1) || M > kSkinnyMaxM) {
      if (why) *why = "skinny plan needs F16 x E2M1 and M <= 16";
      return false;
    }
    if (plan.n_tile != skinny_cols_per_block() || plan.k_tile != skinny_k_chunk() ||
        plan.split_k != 2 || plan.cta_group != 1) {
      if (why) *why = "skinny plan shape not compiled";
      return false;
    }
    return true;
  }
  if (plan.kernel == DG_KERNEL_GEMV) {
    if (!(dtype_a == DG_F16 && dtype_b == DG_F16) || M > kGemvMaxM) {
      if (why) *why = "GEMV plan needs F16 x F16 and M <= 8";
      return false;
    }
    if (plan.split_k < 1 || plan.k_tile <= 0 || plan.k_tile % 8 != 0 ||
        static_cast<int64_t>(plan.k_tile) * plan.split_k < K) {
      if (why) *why = "GEMV plan: K chunks do not cover K";
      return false;
    }
    return true;
  }
  if (plan.kernel == DG_KERNEL_GEMV_MMA) {
    if (!(dtype_a == DG_F16 && dtype_b == DG_F16) || M < 1 || M > kGemvMmaMaxM) {
      if (why) *why = "warp-MMA GEMV plan needs F16 x F16 and M <= 16";
      return false;
    }
    if (plan.split_k < 1 || plan.k_tile <= 0 || plan.k_tile % 8 != 0 ||
        static_cast<int64_t>(plan.k_tile) * plan.split_k < K) {
      if (why) *why = "warp-MMA GEMV plan: K chunks do not cover K";
      return false;
    }
    return true;
  }
  if (why) *why = "plan has no kernel in this library";
  return false;
}

}  // namespace dg
