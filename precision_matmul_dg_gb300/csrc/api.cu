// C ABI of libdg: argument validation, planning, dispatch and error state.
//
// Interface conventions taken from the "DeepGEMM" articles: a null/failure
// return plus a last-error string (discosf.com/news/5532976, section 3.4 and
// section 5.1 question 3: launches are asynchronous and their errors must be
// checked), and positional GEMM arguments A, B, C, alpha, beta, m, n, k
// (kwkr.cn/news/562171, section 3.2 step 4).
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "dg.h"
#include "internal.h"

namespace dg {
namespace {

// Fixed-size per-thread message buffer: recording an error allocates nothing.
thread_local char g_last_error[512];
std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_timeout_ns{0};
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;

dg_status fail(dg_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return s;
}

dg_status fail_cuda(cudaError_t e, const char* what) {
  return fail(DG_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

struct DeviceState {
  bool ready = false;
  dg_hw_desc hw{};
  int* status = nullptr;  // device status word
};

struct Workspace {
  float* partial = nullptr;
  int64_t partial_elems = 0;
  unsigned* counters = nullptr;
  int64_t counter_elems = 0;
  __half* wide = nullptr;  // FP16 copies of widened int8 / E2M1 operands
  int64_t wide_elems = 0;
  void* table = nullptr;   // problem descriptors of a grouped launch
  int64_t table_bytes = 0;
  float* sk_partial = nullptr;  // stream-K partial tiles
  int64_t sk_partial_elems = 0;
  unsigned* sk_sync = nullptr;  // stream-K epoch, finished-CTA count and flags
  int64_t sk_sync_elems = 0;
};

std::mutex g_mu;
std::map<int, DeviceState> g_devices;
std::map<std::pair<int, cudaStream_t>, Workspace> g_workspaces;

// Device copies of host operands for dg_gemm_host, and the two internal
// streams (with their events) that overlap panel copies with the kernels.
struct HostWorkspace {
  void* buf[4] = {nullptr, nullptr, nullptr, nullptr};  // A, B, C/D, bias
  int64_t bytes[4] = {0, 0, 0, 0};
  cudaStream_t aux[2] = {nullptr, nullptr};
  cudaEvent_t ev_b = nullptr;
  cudaEvent_t ev_done[2] = {nullptr, nullptr};
};
std::map<std::pair<int, cudaStream_t>, HostWorkspace> g_host_ws;
std::map<std::tuple<int, int64_t, int64_t, int64_t, int, int, int>, dg_tile_plan> g_plans;

dg_status fill_hw(int device, dg_hw_desc* out) {
  int count = 0;
  cudaError_t e = cudaGetDeviceCount(&count);
  if (e != cudaSuccess || count == 0) {
    cudaGetLastError();
    return fail(DG_ERR_INVALID_STATE, "no CUDA device available (%s)", cudaGetErrorName(e));
  }
  if (device < 0 || device >= count) return fail(DG_ERR_INVALID_STATE, "no device %d", device);
  auto attr = [&](cudaDeviceAttr a) {
    int v = 0;
    cudaDeviceGetAttribute(&v, a, device);
    return v;
  };
  dg_hw_desc h{};
  h.sm_count = attr(cudaDevAttrMultiProcessorCount);
  h.cc_major = attr(cudaDevAttrComputeCapabilityMajor);
  h.cc_minor = attr(cudaDevAttrComputeCapabilityMinor);
  h.smem_per_block_optin = attr(cudaDevAttrMaxSharedMemoryPerBlockOptin);
  h.smem_per_sm = attr(cudaDevAttrMaxSharedMemoryPerMultiprocessor);
  h.regs_per_sm = attr(cudaDevAttrMaxRegistersPerMultiprocessor);
  h.regs_per_thread_max = 255;
  h.max_threads_per_sm = attr(cudaDevAttrMaxThreadsPerMultiProcessor);
  // Tensor memory (512 columns x 128 lanes per SM) exists on the sm_100 family.
  h.tmem_cols = (h.cc_major == 10) ? 512 : 0;
  h.l2_bytes = attr(cudaDevAttrL2CacheSize);
  const double mem_khz = attr(cudaDevAttrMemoryClockRate);
  const double bus_bits = attr(cudaDevAttrGlobalMemoryBusWidth);
  h.hbm_gbps = mem_khz * 1e3 * 2.0 * bus_bits / 8.0 / 1e9;
  h.clock_ghz = attr(cudaDevAttrClockRate) / 1e6;
  // Dense FP16 tensor rate of an sm_100-family SM: 8192 FLOP per clock.
  h.tc_f16_tflops = (h.cc_major == 10) ? h.sm_count * 8192.0 * h.clock_ghz * 1e9 / 1e12 : 0.0;
  *out = h;
  return DG_OK;
}

dg_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(DG_ERR_INVALID_STATE, "no current CUDA device (%s)", cudaGetErrorName(e));
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_devices[dev];
  if (!st.ready) {
    dg_status s = fill_hw(dev, &st.hw);
    if (s != DG_OK) return s;
    if (st.hw.cc_major != 10 || st.hw.cc_minor != 3) {
      return fail(DG_ERR_INVALID_STATE,
                  "device %d is sm_%d%d; libdg is built for sm_103a (GB300) only", dev,
                  st.hw.cc_major, st.hw.cc_minor);
    }
    e = cudaMalloc(&st.status, sizeof(int));
    if (e != cudaSuccess) return fail_cuda(e, "cudaMalloc(status word)");
    e = cudaMemset(st.status, 0, sizeof(int));
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemset(status word)");
    st.ready = true;
  }
  *out = &st;
  return DG_OK;
}

int elem_bits(dg_dtype t) {
  switch (t) {
    case DG_F16: return 16;
    case DG_I8: return 8;
    case DG_E2M1: return 4;
    case DG_MXF4: return 4;  // codes; the scales are a separate array
  }
  return 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A call's epilogue as the kernels take it: kEpiBias | kEpiGelu for the
// fixed forms, kEpiProgram (+ kEpiBias when an op reads the bias) for a
// program.
struct EpiSpec {
  int flags = 0;
  int n_ops = 0;
  EpiOp ops[kMaxEpiOps] = {};
};

dg_status fixed_epilogue(dg_epilogue e, EpiSpec* out) {
  if (e < DG_EPI_NONE || e > DG_EPI_BIAS_GELU)
    return fail(DG_ERR_INVALID_ARG, "unknown epilogue %d", static_cast<int>(e));
  *out = EpiSpec{};
  out->flags = ((e == DG_EPI_BIAS || e == DG_EPI_BIAS_GELU) ? kEpiBias : 0) |
               ((e == DG_EPI_GELU || e == DG_EPI_BIAS_GELU) ? kEpiGelu : 0);
  return DG_OK;
}

dg_status program_epilogue(const dg_epilogue_program* prog, EpiSpec* out) {
  *out = EpiSpec{};
  if (!prog || prog->n_ops == 0) return DG_OK;
  if (prog->n_ops < 0 || prog->n_ops > kMaxEpiOps)
    return fail(DG_ERR_INVALID_ARG, "epilogue program of %d ops (0 .. %d)", prog->n_ops,
                kMaxEpiOps);
  out->flags = kEpiProgram;
  out->n_ops = prog->n_ops;
  for (int k = 0; k < prog->n_ops; ++k) {
    const dg_epilogue_op& op = prog->ops[k];
    switch (op.type) {
      case DG_OP_BIAS:
        out->flags |= kEpiBias;
        break;
      case DG_OP_RELU:
      case DG_OP_GELU:
        break;
      case DG_OP_SCALE:
        if (!isfinite(op.a)) return fail(DG_ERR_INVALID_ARG, "op %d: scale is not finite", k);
        break;
      case DG_OP_CLAMP:
        if (!(op.a <= op.b)) return fail(DG_ERR_INVALID_ARG, "op %d: clamp needs a <= b", k);
        break;
      case DG_OP_QUANT_I8:
        if (k != prog->n_ops - 1)
          return fail(DG_ERR_INVALID_ARG, "op %d: the int8 quantization must be the last op", k);
        if (!isfinite(op.a))
          return fail(DG_ERR_INVALID_ARG, "op %d: quantization scale is not finite", k);
        out->flags |= kEpiOutI8;
        break;
      default:
        return fail(DG_ERR_INVALID_ARG, "op %d: unknown op type %d", k, op.type);
    }
    out->ops[k] = op;
  }
  return DG_OK;
}

dg_status validate(int64_t M, int64_t N, int64_t K, dg_dtype da, dg_dtype db, const void* A,
                   int64_t lda, const void* B, int64_t ldb, void* D, const void* bias,
                   float alpha, float beta, int epi_flags) {
  const bool pair_ok = (da == DG_F16 && db == DG_F16) || (da == DG_I8 && db == DG_I8) ||
                       (da == DG_F16 && db == DG_E2M1);
  if (!pair_ok)
    return fail(DG_ERR_UNSUPPORTED, "dtype pair (%d, %d) not supported: F16xF16, I8xI8, F16xE2M1",
                static_cast<int>(da), static_cast<int>(db));
  if (M < 0 || N < 0 || K < 0) return fail(DG_ERR_INVALID_ARG, "negative size");
  if (M > (int64_t(1) << 30) || N > (int64_t(1) << 30) || K > (int64_t(1) << 30))
    return fail(DG_ERR_INVALID_ARG, "size above 2^30");
  if (M == 0 || N == 0) return DG_OK;
  if (!D) return fail(DG_ERR_INVALID_ARG, "C/D is null");
  if (!aligned16(D)) return fail(DG_ERR_INVALID_ARG, "C/D is not 16-byte aligned");
  if (da == DG_I8) {
    if (epi_flags != 0)
      return fail(DG_ERR_UNSUPPORTED, "the INT8 path has no bias/GELU epilogue or program");
    if (!(isfinite(alpha) && isfinite(beta)) || alpha != floorf(alpha) || beta != floorf(beta) ||
        fabsf(alpha) >= 2147483648.0f || fabsf(beta) >= 2147483648.0f)
      return fail(DG_ERR_UNSUPPORTED, "the INT8 path takes integral alpha and beta below 2^31");
  } else if (!(isfinite(alpha) && isfinite(beta))) {
    return fail(DG_ERR_INVALID_ARG, "alpha and beta must be finite");
  }
  if (epi_flags & kEpiBias) {
    if (!bias) return fail(DG_ERR_INVALID_ARG, "bias epilogue with a null bias");
    if (reinterpret_cast<uintptr_t>(bias) & 1u)
      return fail(DG_ERR_INVALID_ARG, "bias is not 2-byte aligned");
  }
  if (K == 0) return DG_OK;
  if (!A || !B) return fail(DG_ERR_INVALID_ARG, "A or B is null");
  if (!aligned16(A) || !aligned16(B))
    return fail(DG_ERR_INVALID_ARG, "A and B must be 16-byte aligned");
  if (lda < K) return fail(DG_ERR_INVALID_ARG, "lda (%lld) < K (%lld)", (long long)lda, (long long)K);
  if (ldb < K) return fail(DG_ERR_INVALID_ARG, "ldb (%lld) < K (%lld)", (long long)ldb, (long long)K);
  if ((lda * elem_bits(da)) % 128 != 0)
    return fail(DG_ERR_INVALID_ARG, "lda * element size must be a multiple of 16 bytes");
  if (db == DG_E2M1 && (ldb % 2) != 0) return fail(DG_ERR_INVALID_ARG, "E2M1 ldb must be even");
  if ((ldb * elem_bits(db)) % 128 != 0)
    return fail(DG_ERR_INVALID_ARG, "ldb * element size must be a multiple of 16 bytes");
  return DG_OK;
}

uint64_t timeout_ns() {
  const uint64_t t = g_timeout_ns.load();
  return t ? t : kDefaultTimeoutNs;
}

dg_status get_workspace(int dev, cudaStream_t stream, int64_t partial_elems, int64_t counter_elems,
                        SplitKWorkspace* out) {
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace& w = g_workspaces[std::make_pair(dev, stream)];
  if (w.partial_elems < partial_elems) {
    if (w.partial) cudaFree(w.partial);  // synchronises the device: no kernel still uses it
    w.partial = nullptr;
    w.partial_elems = 0;
    cudaError_t e = cudaMalloc(&w.partial, partial_elems * sizeof(float));
    if (e != cudaSuccess) return fail_cuda(e, "cudaMalloc(split-K partials)");
    w.partial_elems = partial_elems;
  }
  if (w.counter_elems < counter_elems) {
    if (w.counters) cudaFree(w.counters);
    w.counters = nullptr;
    w.counter_elems = 0;
    cudaError_t e = cudaMalloc(&w.counters, counter_elems * sizeof(unsigned));
    if (e != cudaSuccess) return fail_cuda(e, "cudaMalloc(split-K counters)");
    e = cudaMemset(w.counters, 0, counter_elems * sizeof(unsigned));
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemset(split-K counters)");
    w.counter_elems = counter_elems;
  }
  out->partial = w.partial;
  out->partial_elems = w.partial_elems;
  out->counters = w.counters;
  out->counter_elems = w.counter_elems;
  return DG_OK;
}

// Device buffer of at least `bytes` for a grouped launch's problem table (per
// device and stream).
dg_status get_table_workspace(int dev, cudaStream_t stream, int64_t bytes, void** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace& w = g_workspaces[std::make_pair(dev, stream)];
  if (w.table_bytes < bytes) {
    if (w.table) cudaFree(w.table);  // synchronises the device: no kernel still reads it
    w.table = nullptr;
    w.table_bytes = 0;
    const cudaError_t e = cudaMalloc(&w.table, bytes);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMalloc(group table)");
    w.table_bytes = bytes;
  }
  *out = w.table;
  return DG_OK;
}

// FP16 buffer of at least `elems` halves for widened operands (per device and stream).
dg_status get_wide_workspace(int dev, cudaStream_t stream, int64_t elems, __half** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace& w = g_workspaces[std::make_pair(dev, stream)];
  if (w.wide_elems < elems) {
    if (w.wide) cudaFree(w.wide);  // synchronises the device: no kernel still uses it
    w.wide = nullptr;
    w.wide_elems = 0;
    cudaError_t e = cudaMalloc(&w.wide, elems * sizeof(__half));
    if (e != cudaSuccess) return fail_cuda(e, "cudaMalloc(widened operands)");
    w.wide_elems = elems;
  }
  *out = w.wide;
  return DG_OK;
}

dg_status dispatch(const GemmArgs& a, const dg_tile_plan& plan, int dev);

// The planner's best plan for a shape and dtype pair on device `dev`, cached
// (the choice does not depend on the epilogue).  DG_LOG=1 prints each plan.
dg_status cached_plan(int dev, int64_t M, int64_t N, int64_t K, dg_dtype da, dg_dtype db,
                      const dg_hw_desc& hw, dg_tile_plan* out) {
  const auto key = std::make_tuple(dev, M, N, K, static_cast<int>(da), static_cast<int>(db), 0);
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_plans.find(key);
    if (it != g_plans.end()) {
      *out = it->second;
      return DG_OK;
    }
  }
  std::string why;
  int n = 0;
  dg_tile_plan plan{};
  const dg_status s = plan_tiles(M, N, K, da, db, DG_EPI_NONE, hw, 0.0, &plan, 1, &n, &why);
  if (s != DG_OK || n == 0)
    return fail(DG_ERR_NO_VALID_CANDIDATE, "no valid candidate found after pruning: %s",
                why.c_str());
  static const bool log_plans = getenv("DG_LOG") != nullptr;
  if (log_plans) {
    fprintf(stderr,
            "[dg] M=%lld N=%lld K=%lld kernel=%d tile=%dx%dx%d split_k=%d stages=%d grid=%d "
            "est=%.2fus\n",
            (long long)M, (long long)N, (long long)K, plan.kernel, plan.m_tile, plan.n_tile,
            plan.k_tile, plan.split_k, plan.stages, plan.grid, plan.est_us);
  }
  std::lock_guard<std::mutex> lock(g_mu);
  g_plans[key] = plan;
  *out = plan;
  return DG_OK;
}

// Strided batch of one problem shape (dg_gemm_strided_batched): problem z
// at A + z sa, B + z sb, C/D + z sc, bias + z sbias (elements; codes for
// E2M1).  Validated by the caller.
struct BatchSpec {
  int64_t count = 1;
  int64_t sa = 0, sb = 0, sc = 0, sbias = 0;
};

// D (leading dimension ldd) = epilogue(alpha * A.B + beta * C (ldc)), for
// one problem or a strided batch.  The caller has validated the epilogue
// (and the batch strides); C and D are checked here.
dg_status run(int64_t M, int64_t N, int64_t K, dg_dtype da, dg_dtype db, const void* A,
              int64_t lda, const void* B, int64_t ldb, const void* C, int64_t ldc, void* D,
              int64_t ldd, const void* bias, float alpha, float beta, const EpiSpec& epi,
              const dg_tile_plan* forced, cudaStream_t stream,
              const BatchSpec& batch = BatchSpec()) {
  dg_status s = validate(M, N, K, da, db, A, lda, B, ldb, D, bias, alpha, beta, epi.flags);
  if (s != DG_OK) return s;
  if (M == 0 || N == 0) return DG_OK;
  if (ldd < N) return fail(DG_ERR_INVALID_ARG, "ldd (%lld) < N (%lld)", (long long)ldd, (long long)N);
  if (beta != 0.0f) {
    if (!C) return fail(DG_ERR_INVALID_ARG, "beta != 0 with a null C");
    if (!aligned16(C)) return fail(DG_ERR_INVALID_ARG, "C is not 16-byte aligned");
    if (ldc < N)
      return fail(DG_ERR_INVALID_ARG, "ldc (%lld) < N (%lld)", (long long)ldc, (long long)N);
    if (C == D && ldc != ldd)
      return fail(DG_ERR_INVALID_ARG, "C and D share a buffer with ldc != ldd");
    if (C == D && (epi.flags & kEpiOutI8))
      return fail(DG_ERR_INVALID_ARG, "an int8 D cannot also be the FP16 C");
  } else {
    C = D;  // never read
    ldc = ldd;
  }
  DeviceState* st = nullptr;
  s = device_state(&st);
  if (s != DG_OK) return s;
  int dev = 0;
  cudaGetDevice(&dev);

  GemmArgs a;
  a.M = M;
  a.N = N;
  a.K = K;
  a.dtype_a = da;
  a.dtype_b = db;
  a.A = A;
  a.lda = lda;
  a.B = B;
  a.ldb = ldb;
  a.C = C;
  a.ldc = ldc;
  a.D = D;
  a.ldd = ldd;
  a.bias = bias;
  a.alpha = alpha;
  a.beta = beta;
  a.epi = epi.flags;
  a.n_ops = epi.n_ops;
  for (int k = 0; k < kMaxEpiOps; ++k) a.ops[k] = epi.ops[k];
  a.stream = stream;
  a.status = st->status;
  a.timeout_ns = timeout_ns();
  a.sm_count = st->hw.sm_count;
  a.exact_i32 = false;
  a.batch = 1;
  a.stride_a = a.stride_b = a.stride_c = a.stride_d = a.stride_bias = 0;

  // Problem z of the batch as a single problem.
  const int64_t out_bytes = da == DG_I8 ? 4 : 2;
  auto problem = [&](int64_t z) {
    GemmArgs w = a;
    w.A = static_cast<const uint8_t*>(A) + z * batch.sa * elem_bits(da) / 8;
    w.B = static_cast<const uint8_t*>(B) + z * batch.sb * elem_bits(db) / 8;
    w.C = static_cast<const uint8_t*>(C) + z * batch.sc * out_bytes;
    w.D = static_cast<uint8_t*>(D) + z * batch.sc * out_bytes;
    w.bias = bias ? static_cast<const uint8_t*>(bias) + z * batch.sbias * 2 : nullptr;
    return w;
  };

  if (K == 0) {
    for (int64_t z = 0; z < batch.count; ++z) {
      cudaError_t e = launch_epilogue_only(problem(z));
      if (e != cudaSuccess) return fail_cuda(e, "epilogue-only launch");
    }
    return DG_OK;
  }

  dg_tile_plan plan{};
  if (forced) {
    std::string why;
    if (!plan_is_runnable(*forced, M, N, K, da, db, &why))
      return fail(DG_ERR_INVALID_STATE, "plan not runnable: %s", why.c_str());
    plan = *forced;
  } else {
    s = cached_plan(dev, M, N, K, da, db, st->hw, &plan);
    if (s != DG_OK) return s;
  }

  if (plan.kernel == DG_KERNEL_GEMV || plan.kernel == DG_KERNEL_GEMV_MMA) {
    // The GEMV kernels take the whole batch in one launch (grid.z).
    const bool mma = plan.kernel == DG_KERNEL_GEMV_MMA;
    if (batch.count > 1 && !forced) {
      int64_t chunk = 0;
      plan.split_k = mma ? gemv_mma_best_split(M, N, K, st->hw, &chunk, batch.count)
                         : gemv_best_split(M, N, K, st->hw, &chunk, batch.count);
      plan.k_tile = static_cast<int>(chunk);
    }
    SplitKWorkspace ws{nullptr, 0, nullptr, 0};
    if (plan.split_k > 1) {
      s = get_workspace(dev, stream, gemv_partial_elems(plan, M, N, batch.count),
                        gemv_counter_elems(plan, N, batch.count), &ws);
      if (s != DG_OK) return s;
    }
    a.batch = batch.count;
    a.stride_a = batch.sa;
    a.stride_b = batch.sb;
    a.stride_c = batch.sc;
    a.stride_d = batch.sc;
    a.stride_bias = batch.sbias;
    const cudaError_t e = mma ? launch_gemv_mma(a, plan, ws) : launch_gemv(a, plan, ws);
    return e == cudaSuccess ? DG_OK : fail_cuda(e, "kernel launch");
  }
  // Other kernels: one launch (or widening + launch) per problem.
  for (int64_t z = 0; z < batch.count; ++z) {
    s = dispatch(problem(z), plan, dev);
    if (s != DG_OK) return s;
  }
  return DG_OK;
}

// Launches `plan` (not the GEMV) for the single problem `a`.
dg_status dispatch(const GemmArgs& a, const dg_tile_plan& plan, int dev) {
  const int64_t M = a.M, N = a.N, K = a.K;
  const dg_dtype da = a.dtype_a, db = a.dtype_b;
  const cudaStream_t stream = a.stream;
  dg_status s = DG_OK;
  cudaError_t e = cudaSuccess;
  if (plan.kernel == DG_KERNEL_SKINNY) {
    e = launch_skinny(a, plan);
  } else if (plan.kernel == DG_KERNEL_TC && da == DG_MXF4) {
    // MXFP4 on the block-scaled MMA: the codes go to the tensor cores as
    // they are, and the kernel loads the scale bytes with TMA, 16 bytes of a
    // row at a time, so each operand's scale rows must start on 16-byte
    // boundaries.  Other scale layouts are first copied into the workspace
    // with a 16-byte row pitch.
    GemmArgs w = a;
    const int64_t nblk = (K + 31) / 32, pitch = (nblk + 15) / 16 * 16;
    const bool fit_a = (reinterpret_cast<uintptr_t>(a.scale_a) & 15) == 0 && a.lds_a % 16 == 0;
    const bool fit_b = (reinterpret_cast<uintptr_t>(a.scale_b) & 15) == 0 && a.lds_b % 16 == 0;
    if (!fit_a || !fit_b) {
      const int64_t bytes = (fit_a ? 0 : M * pitch) + (fit_b ? 0 : N * pitch);
      __half* ws = nullptr;
      s = get_wide_workspace(dev, stream, (bytes + 1) / 2, &ws);
      if (s != DG_OK) return s;
      uint8_t* dst = reinterpret_cast<uint8_t*>(ws);
      if (!fit_a) {
        e = cudaMemcpy2DAsync(dst, pitch, a.scale_a, a.lds_a, nblk, M, cudaMemcpyDeviceToDevice,
                              stream);
        if (e != cudaSuccess) return fail_cuda(e, "scale copy");
        w.scale_a = dst;
        w.lds_a = pitch;
        dst += M * pitch;
      }
      if (!fit_b) {
        e = cudaMemcpy2DAsync(dst, pitch, a.scale_b, a.lds_b, nblk, N, cudaMemcpyDeviceToDevice,
                              stream);
        if (e != cudaSuccess) return fail_cuda(e, "scale copy");
        w.scale_b = dst;
        w.lds_b = pitch;
      }
    }
    e = launch_tc_mx(w, plan);
  } else if (plan.kernel == DG_KERNEL_TC && plan.swap_ab) {
    // FP16 x E2M1 with the weights widened in tensor memory.  Layouts its
    // TMA copies cannot take run the widening path on a compiled FP16 tile.
    if (!w4t_layout_ok(a)) {
      dg_tile_plan wp = plan;
      wp.kernel = DG_KERNEL_TC_WIDENED;
      wp.swap_ab = 0;
      wp.k_tile = 64;
      wp.split_k = 1;
      wp.grid = 0;
      wp.cta_group = M > 128 ? 2 : 1;
      wp.m_tile = 128 * wp.cta_group;
      wp.n_tile = M > 128 ? 192 : 128;
      wp.stages = 6;
      return dispatch(a, wp, dev);
    }
    e = launch_w4t(a, plan);
  } else if (plan.kernel == DG_KERNEL_TC) {
    e = (da == DG_F16 && db == DG_F16) ? launch_tc(a, plan) : launch_conv(a, plan);
  } else if (plan.kernel == DG_KERNEL_TC_STREAMK) {
    e = launch_tc_streamk(a, plan);
  } else if (plan.kernel == DG_KERNEL_TC_WIDENED && da == DG_MXF4) {
    // Widen both MXFP4 operands with their block scales into BF16 copies
    // (exact), then the tensor-core kernel on BF16 operands.
    const int64_t ldw = widened_ld(K);
    __half* wide = nullptr;
    s = get_wide_workspace(dev, stream, (M + N) * ldw, &wide);
    if (s != DG_OK) return s;
    const MxWidenJob jobs[2] = {{a.A, M, a.lda, a.scale_a, a.lds_a, wide},
                                {a.B, N, a.ldb, a.scale_b, a.lds_b, wide + M * ldw}};
    e = launch_widen_mxf4(jobs, 2, K, stream, a.sm_count);
    if (e != cudaSuccess) return fail_cuda(e, "widening launch");
    GemmArgs w = a;
    w.A = wide;
    w.lda = ldw;
    w.B = wide + M * ldw;
    w.ldb = ldw;
    w.dtype_a = DG_F16;
    w.dtype_b = DG_F16;
    w.bf16_ab = true;
    e = launch_tc(w, plan);
  } else if (plan.kernel == DG_KERNEL_TC_WIDENED) {
    // Widen the narrow operands into FP16 copies, then the FP16 kernel.
    const int64_t ldw = widened_ld(K);
    const int64_t a_elems = da == DG_I8 ? M * ldw : 0;
    __half* wide = nullptr;
    s = get_wide_workspace(dev, stream, a_elems + N * ldw, &wide);
    if (s != DG_OK) return s;
    GemmArgs w = a;
    WidenJob jobs[2];
    int njobs = 0;
    if (da == DG_I8) {
      jobs[njobs++] = WidenJob{DG_I8, a.A, M, a.lda, wide};
      w.A = wide;
      w.lda = ldw;
    }
    jobs[njobs++] = WidenJob{db, a.B, N, a.ldb, wide + a_elems};
    e = launch_widen(jobs, njobs, K, stream, a.sm_count);
    if (e != cudaSuccess) return fail_cuda(e, "widening launch");
    w.B = wide + a_elems;
    w.ldb = ldw;
    w.dtype_a = DG_F16;
    w.dtype_b = DG_F16;
    w.exact_i32 = da == DG_I8;
    e = launch_tc(w, plan);
  } else {
    return fail(DG_ERR_INVALID_STATE, "plan names no kernel of this library");
  }
  if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
  return DG_OK;
}

// Rules shared by the MXFP4 entry points for one packed operand: rows of
// `ld` codes (>= K, a multiple of 32, so 16-byte rows) at a 16-byte aligned
// base, and `lds` >= ceil(K / 32) scale bytes per row.
dg_status check_mx_operand(const char* name, int64_t K, const void* codes, int64_t ld,
                           const void* scales, int64_t lds) {
  if (!codes || !scales) return fail(DG_ERR_INVALID_ARG, "%s or its scales is null", name);
  if (!aligned16(codes)) return fail(DG_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  if (ld < K || ld % 32 != 0)
    return fail(DG_ERR_INVALID_ARG,
                "%s: leading dimension %lld codes must be >= K (%lld) and a multiple of 32", name,
                (long long)ld, (long long)K);
  if (lds < (K + 31) / 32)
    return fail(DG_ERR_INVALID_ARG, "%s: %lld scale bytes per row, need %lld", name,
                (long long)lds, (long long)((K + 31) / 32));
  return DG_OK;
}

// dg_quantize_mxf4 (dg.h).
dg_status run_quantize_mxf4(int64_t rows, int64_t K, const void* X, int64_t ldx, void* codes,
                            int64_t ldq, void* scales, int64_t lds, cudaStream_t stream) {
  if (rows < 0 || K < 0) return fail(DG_ERR_INVALID_ARG, "negative size");
  if (rows > (int64_t(1) << 30) || K > (int64_t(1) << 30))
    return fail(DG_ERR_INVALID_ARG, "size above 2^30");
  if (rows == 0 || K == 0) return DG_OK;
  if (!X) return fail(DG_ERR_INVALID_ARG, "X is null");
  if (!aligned16(X) || ldx % 8 != 0 || ldx < K)
    return fail(DG_ERR_INVALID_ARG,
                "X must be 16-byte aligned with ldx >= K and ldx a multiple of 8 elements");
  dg_status s = check_mx_operand("the codes", K, codes, ldq, scales, lds);
  if (s != DG_OK) return s;
  DeviceState* st = nullptr;
  s = device_state(&st);
  if (s != DG_OK) return s;
  const cudaError_t e =
      launch_quantize_mxf4(rows, K, X, ldx, codes, ldq, scales, lds, stream, st->hw.sm_count);
  return e == cudaSuccess ? DG_OK : fail_cuda(e, "quantization launch");
}

// dg_gemm_mxf4 (dg.h): C and D one buffer of leading dimension N.
dg_status run_gemm_mxf4(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                        const void* scale_a, int64_t lds_a, const void* B, int64_t ldb,
                        const void* scale_b, int64_t lds_b, void* C, const void* bias,
                        float alpha, float beta, dg_epilogue epilogue, const dg_tile_plan* forced,
                        cudaStream_t stream) {
  EpiSpec epi;
  dg_status s = fixed_epilogue(epilogue, &epi);
  if (s != DG_OK) return s;
  if (M < 0 || N < 0 || K < 0) return fail(DG_ERR_INVALID_ARG, "negative size");
  if (M > (int64_t(1) << 30) || N > (int64_t(1) << 30) || K > (int64_t(1) << 30))
    return fail(DG_ERR_INVALID_ARG, "size above 2^30");
  if (M == 0 || N == 0) return DG_OK;
  if (!C) return fail(DG_ERR_INVALID_ARG, "C/D is null");
  if (!aligned16(C)) return fail(DG_ERR_INVALID_ARG, "C/D is not 16-byte aligned");
  if (!(isfinite(alpha) && isfinite(beta)))
    return fail(DG_ERR_INVALID_ARG, "alpha and beta must be finite");
  if (epi.flags & kEpiBias) {
    if (!bias) return fail(DG_ERR_INVALID_ARG, "bias epilogue with a null bias");
    if (reinterpret_cast<uintptr_t>(bias) & 1u)
      return fail(DG_ERR_INVALID_ARG, "bias is not 2-byte aligned");
  }
  if (K > 0) {
    if ((s = check_mx_operand("A", K, A, lda, scale_a, lds_a)) != DG_OK) return s;
    if ((s = check_mx_operand("B", K, B, ldb, scale_b, lds_b)) != DG_OK) return s;
  }
  DeviceState* st = nullptr;
  s = device_state(&st);
  if (s != DG_OK) return s;
  int dev = 0;
  cudaGetDevice(&dev);

  GemmArgs a;
  a.M = M;
  a.N = N;
  a.K = K;
  a.dtype_a = DG_MXF4;
  a.dtype_b = DG_MXF4;
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
  a.epi = epi.flags;
  a.n_ops = 0;
  for (int k = 0; k < kMaxEpiOps; ++k) a.ops[k] = EpiOp{};
  a.batch = 1;
  a.stride_a = a.stride_b = a.stride_c = a.stride_d = a.stride_bias = 0;
  a.stream = stream;
  a.status = st->status;
  a.timeout_ns = timeout_ns();
  a.sm_count = st->hw.sm_count;
  a.exact_i32 = false;
  a.scale_a = scale_a;
  a.lds_a = lds_a;
  a.scale_b = scale_b;
  a.lds_b = lds_b;
  if (K == 0) {
    const cudaError_t e = launch_epilogue_only(a);
    return e == cudaSuccess ? DG_OK : fail_cuda(e, "epilogue-only launch");
  }
  dg_tile_plan plan{};
  if (forced) {
    std::string why;
    if (!plan_is_runnable(*forced, M, N, K, DG_MXF4, DG_MXF4, &why))
      return fail(DG_ERR_INVALID_STATE, "plan not runnable: %s", why.c_str());
    plan = *forced;
  } else {
    s = cached_plan(dev, M, N, K, DG_MXF4, DG_MXF4, st->hw, &plan);
    if (s != DG_OK) return s;
  }
  return dispatch(a, plan, dev);
}

}  // namespace

dg_status get_sk_workspace(int dev, cudaStream_t stream, int64_t partial_elems,
                           int64_t sync_elems, float** partial, unsigned** sync) {
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace& w = g_workspaces[std::make_pair(dev, stream)];
  if (w.sk_partial_elems < partial_elems) {
    if (w.sk_partial) cudaFree(w.sk_partial);  // synchronises the device: no kernel still uses it
    w.sk_partial = nullptr;
    w.sk_partial_elems = 0;
    cudaError_t e = cudaMalloc(&w.sk_partial, partial_elems * sizeof(float));
    if (e != cudaSuccess) return fail_cuda(e, "cudaMalloc(stream-K partials)");
    w.sk_partial_elems = partial_elems;
  }
  if (w.sk_sync_elems < sync_elems) {
    if (w.sk_sync) cudaFree(w.sk_sync);
    w.sk_sync = nullptr;
    w.sk_sync_elems = 0;
    cudaError_t e = cudaMalloc(&w.sk_sync, sync_elems * sizeof(unsigned));
    if (e != cudaSuccess) return fail_cuda(e, "cudaMalloc(stream-K flags)");
    // epoch 0, no CTA finished, no flag raised
    e = cudaMemset(w.sk_sync, 0, sync_elems * sizeof(unsigned));
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemset(stream-K flags)");
    w.sk_sync_elems = sync_elems;
  }
  *partial = w.sk_partial;
  *sync = w.sk_sync;
  return DG_OK;
}

void count_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n)); }

void clear_error() { g_last_error[0] = '\0'; }

dg_status set_error(dg_status s, const char* msg) { return fail(s, "%s", msg); }

// Host-buffer GEMM (dg_gemm_host in dg.h).
dg_status run_host(int64_t M, int64_t N, int64_t K, dg_dtype da, dg_dtype db, const void* A,
                   int64_t lda, const void* B, int64_t ldb, const void* C, void* D,
                   const void* bias, float alpha, float beta, dg_epilogue epilogue,
                   cudaStream_t stream) {
  clear_error();
  if (!D) return fail(DG_ERR_INVALID_ARG, "D is null");
  if (beta != 0.0f && !C) return fail(DG_ERR_INVALID_ARG, "beta != 0 with a null C");
  EpiSpec epi;
  dg_status s = fixed_epilogue(epilogue, &epi);
  if (s != DG_OK) return s;
  s = validate(M, N, K, da, db, A, lda, B, ldb, D, bias, alpha, beta, epi.flags);
  if (s != DG_OK) return s;
  if (M == 0 || N == 0) return DG_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return fail(DG_ERR_INVALID_STATE, "no current CUDA device");
  }
  const int64_t a_row = lda * elem_bits(da) / 8, b_row = ldb * elem_bits(db) / 8;
  const int64_t o_elem = da == DG_I8 ? 4 : 2;
  const bool has_bias = epilogue == DG_EPI_BIAS || epilogue == DG_EPI_BIAS_GELU;
  const int64_t need[4] = {K > 0 ? M * a_row : 0, K > 0 ? N * b_row : 0, M * N * o_elem,
                           has_bias ? N * 2 : 0};
  HostWorkspace* hw = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    hw = &g_host_ws[std::make_pair(dev, stream)];
    for (int i = 0; i < 4; ++i) {
      if (hw->bytes[i] >= need[i]) continue;
      if (hw->buf[i]) cudaFree(hw->buf[i]);  // synchronises the device: nothing still uses it
      hw->buf[i] = nullptr;
      hw->bytes[i] = 0;
      const cudaError_t e = cudaMalloc(&hw->buf[i], need[i]);
      if (e != cudaSuccess) return fail_cuda(e, "cudaMalloc(host-call workspace)");
      hw->bytes[i] = need[i];
    }
    if (!hw->aux[0]) {
      for (int i = 0; i < 2; ++i) {
        cudaError_t e = cudaStreamCreateWithFlags(&hw->aux[i], cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hw->ev_done[i], cudaEventDisableTiming);
        if (e != cudaSuccess) return fail_cuda(e, "stream / event creation");
      }
      const cudaError_t e = cudaEventCreateWithFlags(&hw->ev_b, cudaEventDisableTiming);
      if (e != cudaSuccess) return fail_cuda(e, "event creation");
    }
  }
  auto* dA = static_cast<uint8_t*>(hw->buf[0]);
  auto* dB = static_cast<uint8_t*>(hw->buf[1]);
  auto* dC = static_cast<uint8_t*>(hw->buf[2]);
  auto* dbias = static_cast<uint8_t*>(hw->buf[3]);
  auto copy = [&](void* dst, const void* src, int64_t n, cudaMemcpyKind kind,
                  cudaStream_t st) -> dg_status {
    if (n <= 0) return DG_OK;
    const cudaError_t e = cudaMemcpyAsync(dst, src, n, kind, st);
    return e == cudaSuccess ? DG_OK : fail_cuda(e, "host-call copy");
  };
  // B and bias first, on the caller's stream (after whatever it already holds).
  if ((s = copy(dB, B, need[1], cudaMemcpyHostToDevice, stream)) != DG_OK) return s;
  if ((s = copy(dbias, bias, need[3], cudaMemcpyHostToDevice, stream)) != DG_OK) return s;
  cudaError_t e = cudaEventRecord(hw->ev_b, stream);
  if (e != cudaSuccess) return fail_cuda(e, "event record");
  // Row panels of A and C: copy in, multiply, copy out, alternating between
  // the two internal streams so that one panel's copies overlap the other's.
  const int64_t panel = M >= 512 ? (((M + 3) / 4 + 255) / 256) * 256 : M;
  const int64_t npanels = (M + panel - 1) / panel;
  for (int64_t i = 0; i < npanels; ++i) {
    cudaStream_t st = hw->aux[i % 2];
    if (i < 2 && (e = cudaStreamWaitEvent(st, hw->ev_b, 0)) != cudaSuccess)
      return fail_cuda(e, "stream wait");
    const int64_t r0 = i * panel, mr = std::min(panel, M - r0);
    if ((s = copy(dA + r0 * a_row, static_cast<const uint8_t*>(A) + r0 * a_row, mr * a_row,
                  cudaMemcpyHostToDevice, st)) != DG_OK)
      return s;
    if (beta != 0.0f &&
        (s = copy(dC + r0 * N * o_elem, static_cast<const uint8_t*>(C) + r0 * N * o_elem,
                  mr * N * o_elem, cudaMemcpyHostToDevice, st)) != DG_OK)
      return s;
    uint8_t* cd = dC + r0 * N * o_elem;
    s = run(mr, N, K, da, db, dA + r0 * a_row, lda, dB, ldb, cd, N, cd, N,
            has_bias ? dbias : nullptr, alpha, beta, epi, nullptr, st);
    if (s != DG_OK) return s;
    if ((s = copy(static_cast<uint8_t*>(D) + r0 * N * o_elem, dC + r0 * N * o_elem,
                  mr * N * o_elem, cudaMemcpyDeviceToHost, st)) != DG_OK)
      return s;
  }
  // The caller's stream continues after both internal streams.
  for (int i = 0; i < 2 && i < npanels; ++i) {
    if ((e = cudaEventRecord(hw->ev_done[i], hw->aux[i])) != cudaSuccess ||
        (e = cudaStreamWaitEvent(stream, hw->ev_done[i], 0)) != cudaSuccess)
      return fail_cuda(e, "stream join");
  }
  return DG_OK;
}

dg_status fill_hw_desc(int device, dg_hw_desc* out) { return fill_hw(device, out); }

dg_status validate_gemm_args(int64_t M, int64_t N, int64_t K, dg_dtype da, dg_dtype db,
                             const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                             const void* bias, float alpha, float beta, dg_epilogue epi) {
  EpiSpec e;
  const dg_status s = fixed_epilogue(epi, &e);
  if (s != DG_OK) return s;
  return validate(M, N, K, da, db, A, lda, B, ldb, C, bias, alpha, beta, e.flags);
}

}  // namespace dg

using namespace dg;

extern "C" {

dg_status dg_query_hw(int device, dg_hw_desc* out) {
  clear_error();
  if (!out) return fail(DG_ERR_INVALID_ARG, "out is null");
  return fill_hw(device, out);
}

dg_status dg_plan_tiles(int64_t M, int64_t N, int64_t K, dg_dtype dtype_a, dg_dtype dtype_b,
                        dg_epilogue epilogue, const dg_hw_desc* hw, double target_occupancy,
                        dg_tile_plan* out, int max_out, int* n_out) {
  clear_error();
  if (n_out) *n_out = 0;
  if (M <= 0 || N <= 0 || K <= 0) return fail(DG_ERR_INVALID_ARG, "M, N and K must be >= 1");
  if (max_out > 0 && !out) return fail(DG_ERR_INVALID_ARG, "out is null");
  if (!(target_occupancy >= 0.0 && target_occupancy <= 1.0))
    return fail(DG_ERR_INVALID_ARG, "target_occupancy must lie in [0, 1]");
  const bool pair_ok = (dtype_a == DG_F16 && dtype_b == DG_F16) ||
                       (dtype_a == DG_I8 && dtype_b == DG_I8) ||
                       (dtype_a == DG_F16 && dtype_b == DG_E2M1) ||
                       (dtype_a == DG_MXF4 && dtype_b == DG_MXF4);
  if (!pair_ok) return fail(DG_ERR_UNSUPPORTED, "dtype pair not supported");
  dg_hw_desc local{};
  if (!hw) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
      cudaGetLastError();
      return fail(DG_ERR_INVALID_STATE, "hw is null and there is no current CUDA device");
    }
    dg_status s = fill_hw(dev, &local);
    if (s != DG_OK) return s;
    hw = &local;
  }
  if (hw->sm_count <= 0 || hw->smem_per_block_optin <= 0 || hw->regs_per_sm <= 0 ||
      hw->max_threads_per_sm <= 0)
    return fail(DG_ERR_INVALID_ARG, "hardware description has empty fields");
  std::string why;
  dg_status s = plan_tiles(M, N, K, dtype_a, dtype_b, epilogue, *hw, target_occupancy, out,
                           max_out, n_out, &why);
  if (s == DG_ERR_NO_VALID_CANDIDATE)
    return fail(s, "no valid candidate found after pruning: %s", why.c_str());
  return s;
}

dg_status dg_gemm_host(int64_t M, int64_t N, int64_t K, dg_dtype dtype_a, dg_dtype dtype_b,
                       const void* A, int64_t lda, const void* B, int64_t ldb, const void* C,
                       void* D, const void* bias, float alpha, float beta,
                       dg_epilogue epilogue, dg_stream_t stream) {
  return run_host(M, N, K, dtype_a, dtype_b, A, lda, B, ldb, C, D, bias, alpha, beta, epilogue,
                  reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_gemm(int64_t M, int64_t N, int64_t K, dg_dtype dtype_a, dg_dtype dtype_b,
                  const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                  const void* bias, float alpha, float beta, dg_epilogue epilogue,
                  dg_stream_t stream) {
  clear_error();
  EpiSpec epi;
  const dg_status s = fixed_epilogue(epilogue, &epi);
  if (s != DG_OK) return s;
  return run(M, N, K, dtype_a, dtype_b, A, lda, B, ldb, C, N, C, N, bias, alpha, beta, epi,
             nullptr, reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_gemm_ex(int64_t M, int64_t N, int64_t K, dg_dtype dtype_a, dg_dtype dtype_b,
                     const void* A, int64_t lda, const void* B, int64_t ldb, const void* C,
                     int64_t ldc, void* D, int64_t ldd, const void* bias, float alpha, float beta,
                     const dg_epilogue_program* program, dg_stream_t stream) {
  clear_error();
  EpiSpec epi;
  const dg_status s = program_epilogue(program, &epi);
  if (s != DG_OK) return s;
  return run(M, N, K, dtype_a, dtype_b, A, lda, B, ldb, C, ldc, D, ldd, bias, alpha, beta, epi,
             nullptr, reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_gemm_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K,
                                  dg_dtype dtype_a, dg_dtype dtype_b, const void* A, int64_t lda,
                                  int64_t stride_a, const void* B, int64_t ldb, int64_t stride_b,
                                  void* C, int64_t stride_c, const void* bias,
                                  int64_t stride_bias, float alpha, float beta,
                                  dg_epilogue epilogue, dg_stream_t stream) {
  clear_error();
  EpiSpec epi;
  dg_status s = fixed_epilogue(epilogue, &epi);
  if (s != DG_OK) return s;
  if (batch < 0) return fail(DG_ERR_INVALID_ARG, "negative batch");
  if (batch == 0) return DG_OK;
  if (stride_a < 0 || stride_b < 0 || stride_c < 0 || stride_bias < 0)
    return fail(DG_ERR_INVALID_ARG, "negative batch stride");
  if (batch > 1) {
    if (M > 0 && N > 0 && stride_c < M * N)
      return fail(DG_ERR_INVALID_ARG, "stride_c (%lld) < M * N: the problems' outputs overlap",
                  (long long)stride_c);
    if ((stride_a * elem_bits(dtype_a)) % 128 != 0 || (stride_b * elem_bits(dtype_b)) % 128 != 0)
      return fail(DG_ERR_INVALID_ARG, "stride_a and stride_b must span multiples of 16 bytes");
  }
  BatchSpec bs;
  bs.count = batch;
  bs.sa = stride_a;
  bs.sb = stride_b;
  bs.sc = stride_c;
  bs.sbias = stride_bias;
  return run(M, N, K, dtype_a, dtype_b, A, lda, B, ldb, C, N, C, N, bias, alpha, beta, epi,
             nullptr, reinterpret_cast<cudaStream_t>(stream), bs);
}

dg_status dg_gemm_grouped(int64_t count, const int64_t* Ms, int64_t N, int64_t K,
                          dg_dtype dtype_a, dg_dtype dtype_b, const void* const* A, int64_t lda,
                          const void* const* B, int64_t ldb, void* const* C,
                          const void* const* bias, float alpha, float beta,
                          dg_epilogue epilogue, dg_stream_t stream) {
  clear_error();
  EpiSpec epi;
  dg_status s = fixed_epilogue(epilogue, &epi);
  if (s != DG_OK) return s;
  if (count < 0) return fail(DG_ERR_INVALID_ARG, "negative count");
  if (count == 0) return DG_OK;
  if (!Ms || !A || !B || !C)
    return fail(DG_ERR_INVALID_ARG, "Ms, A, B and C must be host arrays of count entries");
  if ((epi.flags & kEpiBias) && !bias)
    return fail(DG_ERR_INVALID_ARG, "bias epilogue with a null bias array");
  int64_t max_m = 0;
  for (int64_t g = 0; g < count; ++g) {
    if (Ms[g] < 0) return fail(DG_ERR_INVALID_ARG, "problem %lld: negative M", (long long)g);
    max_m = std::max(max_m, Ms[g]);
  }
  for (int64_t g = 0; g < count; ++g) {
    if (Ms[g] == 0) continue;
    s = validate(Ms[g], N, K, dtype_a, dtype_b, A[g], lda, B[g], ldb, C[g],
                 bias ? bias[g] : nullptr, alpha, beta, epi.flags);
    if (s != DG_OK) {
      std::string msg = g_last_error;
      return fail(s, "problem %lld: %s", (long long)g, msg.c_str());
    }
  }
  if (max_m == 0 || N == 0) return DG_OK;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool one_launch = dtype_a == DG_F16 && dtype_b == DG_F16 && max_m <= 16 && K > 0;
  if (!one_launch) {  // each problem in turn, as dg_gemm
    for (int64_t g = 0; g < count; ++g) {
      if (Ms[g] == 0) continue;
      s = run(Ms[g], N, K, dtype_a, dtype_b, A[g], lda, B[g], ldb, C[g], N, C[g], N,
              bias ? bias[g] : nullptr, alpha, beta, epi, nullptr, st);
      if (s != DG_OK) return s;
    }
    return DG_OK;
  }
  DeviceState* dst = nullptr;
  s = device_state(&dst);
  if (s != DG_OK) return s;
  int dev = 0;
  cudaGetDevice(&dev);
  // One launch of the warp-MMA GEMV over the group: split-K chosen for the
  // whole group, problem descriptors in a device table.
  dg_tile_plan plan{};
  int64_t chunk = 0;
  plan.kernel = DG_KERNEL_GEMV_MMA;
  plan.split_k = gemv_mma_best_split(max_m, N, K, dst->hw, &chunk, count);
  plan.k_tile = static_cast<int>(chunk);
  SplitKWorkspace ws{nullptr, 0, nullptr, 0};
  if (plan.split_k > 1) {
    s = get_workspace(dev, st, static_cast<int64_t>(plan.split_k) * max_m * N * count,
                      (N + 7) / 8 * count, &ws);
    if (s != DG_OK) return s;
  }
  const int64_t entry = gemv_group_entry_bytes();
  void* table = nullptr;
  s = get_table_workspace(dev, st, entry * count, &table);
  if (s != DG_OK) return s;
  std::vector<unsigned char> host(static_cast<size_t>(entry * count));
  for (int64_t g = 0; g < count; ++g)
    gemv_group_entry(host.data(), g, A[g], B[g], C[g], bias ? bias[g] : nullptr, Ms[g]);
  // From pageable memory the call returns once `host` has been staged; the
  // copy runs in stream order, after the kernels that read the table before.
  cudaError_t e = cudaMemcpyAsync(table, host.data(), host.size(), cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return fail_cuda(e, "group table copy");
  GemmArgs a{};
  a.M = max_m;
  a.N = N;
  a.K = K;
  a.dtype_a = dtype_a;
  a.dtype_b = dtype_b;
  a.lda = lda;
  a.ldb = ldb;
  a.ldc = N;
  a.ldd = N;
  a.alpha = alpha;
  a.beta = beta;
  a.epi = epi.flags;
  a.n_ops = 0;
  a.batch = count;
  a.stream = st;
  a.status = dst->status;
  a.timeout_ns = timeout_ns();
  a.sm_count = dst->hw.sm_count;
  e = launch_gemv_mma_grouped(a, table, count, max_m, plan, ws);
  return e == cudaSuccess ? DG_OK : fail_cuda(e, "kernel launch");
}

dg_status dg_quantize_mxf4(int64_t rows, int64_t K, const void* X, int64_t ldx, void* codes,
                           int64_t ldq, void* scales, int64_t lds, dg_stream_t stream) {
  clear_error();
  return run_quantize_mxf4(rows, K, X, ldx, codes, ldq, scales, lds,
                           reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_gemm_mxf4(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                       const void* scale_a, int64_t lds_a, const void* B, int64_t ldb,
                       const void* scale_b, int64_t lds_b, void* C, const void* bias, float alpha,
                       float beta, dg_epilogue epilogue, dg_stream_t stream) {
  clear_error();
  return run_gemm_mxf4(M, N, K, A, lda, scale_a, lds_a, B, ldb, scale_b, lds_b, C, bias, alpha,
                       beta, epilogue, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_gemm_mxf4_planned(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                               const void* scale_a, int64_t lds_a, const void* B, int64_t ldb,
                               const void* scale_b, int64_t lds_b, void* C, const void* bias,
                               float alpha, float beta, dg_epilogue epilogue,
                               const dg_tile_plan* plan, dg_stream_t stream) {
  clear_error();
  if (!plan) return fail(DG_ERR_INVALID_ARG, "plan is null");
  return run_gemm_mxf4(M, N, K, A, lda, scale_a, lds_a, B, ldb, scale_b, lds_b, C, bias, alpha,
                       beta, epilogue, plan, reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_gemm_planned(int64_t M, int64_t N, int64_t K, dg_dtype dtype_a, dg_dtype dtype_b,
                          const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                          const void* bias, float alpha, float beta, dg_epilogue epilogue,
                          const dg_tile_plan* plan, dg_stream_t stream) {
  clear_error();
  if (!plan) return fail(DG_ERR_INVALID_ARG, "plan is null");
  EpiSpec epi;
  const dg_status s = fixed_epilogue(epilogue, &epi);
  if (s != DG_OK) return s;
  return run(M, N, K, dtype_a, dtype_b, A, lda, B, ldb, C, N, C, N, bias, alpha, beta, epi, plan,
             reinterpret_cast<cudaStream_t>(stream));
}

const char* dg_last_error(void) { return g_last_error; }

dg_status dg_check_status(dg_stream_t stream) {
  clear_error();
  DeviceState* st = nullptr;
  dg_status s = device_state(&st);
  if (s != DG_OK) return s;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
  int word = 0;
  e = cudaMemcpy(&word, st->status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e, "reading the status word");
  if (word != 0) {
    const int zero = 0;
    cudaMemcpy(st->status, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (word == static_cast<int>(DG_ERR_TIMEOUT))
      return fail(DG_ERR_TIMEOUT, "a kernel gave up on a pipeline wait after its time limit");
    return fail(DG_ERR_INVALID_STATE, "device status word %d", word);
  }
  return DG_OK;
}

dg_status dg_set_wait_timeout_ns(uint64_t ns) {
  clear_error();
  g_timeout_ns.store(ns);
  return DG_OK;
}

dg_status dg_selftest_wait_timeout(dg_stream_t stream) {
  clear_error();
  DeviceState* st = nullptr;
  dg_status s = device_state(&st);
  if (s != DG_OK) return s;
  cudaError_t e = launch_wait_selftest(reinterpret_cast<cudaStream_t>(stream), st->status,
                                       timeout_ns());
  return e == cudaSuccess ? DG_OK : fail_cuda(e, "self-test launch");
}

uint64_t dg_launch_count(void) { return g_launches.load(); }

dg_status dg_shutdown(void) {
  clear_error();
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  const bool have_dev = cudaGetDevice(&cur) == cudaSuccess;
  for (auto& kv : g_workspaces) {
    cudaSetDevice(kv.first.first);
    if (kv.second.partial) cudaFree(kv.second.partial);
    if (kv.second.counters) cudaFree(kv.second.counters);
    if (kv.second.wide) cudaFree(kv.second.wide);
    if (kv.second.table) cudaFree(kv.second.table);
    if (kv.second.sk_partial) cudaFree(kv.second.sk_partial);
    if (kv.second.sk_sync) cudaFree(kv.second.sk_sync);
  }
  g_workspaces.clear();
  for (auto& kv : g_host_ws) {
    cudaSetDevice(kv.first.first);
    HostWorkspace& h = kv.second;
    for (int i = 0; i < 4; ++i)
      if (h.buf[i]) cudaFree(h.buf[i]);
    for (int i = 0; i < 2; ++i) {
      if (h.aux[i]) cudaStreamDestroy(h.aux[i]);
      if (h.ev_done[i]) cudaEventDestroy(h.ev_done[i]);
    }
    if (h.ev_b) cudaEventDestroy(h.ev_b);
  }
  g_host_ws.clear();
  for (auto& kv : g_devices) {
    if (kv.second.status) {
      cudaSetDevice(kv.first);
      cudaFree(kv.second.status);
    }
  }
  g_devices.clear();
  g_plans.clear();
  if (have_dev) cudaSetDevice(cur);
  cudaGetLastError();
  return DG_OK;
}

}  // extern "C"
