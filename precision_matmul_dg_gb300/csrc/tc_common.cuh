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

// v[i] += bias[col0 + i] for the columns < N: four 16-byte loads (the same
// address across the warp) when the 32 values are in range and aligned.
__device__ __forceinline__ void add_bias_chunk(float (&v)[32], const __half* bias, int col0,
                                               int N) {
  const __half* b = bias + col0;
  if (col0 + 32 <= N && (reinterpret_cast<uintptr_t>(b) & 15) == 0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 bv = __ldg(reinterpret_cast<const uint4*>(b) + q);
      const __half2* bh = reinterpret_cast<const __half2*>(&bv);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float2 f = __half22float2(bh[h]);
        v[q * 8 + 2 * h] += f.x;
        v[q * 8 + 2 * h + 1] += f.y;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col0 + i < N) v[i] += __half2float(__ldg(b + i));
  }
}

// An epilogue program's ops, in order, on 32 consecutive columns of one row
// (op-outer, so each op's kind is decided once per chunk, uniformly across
// the warp).  Columns >= N take a zero bias; their values are never stored.
__device__ __forceinline__ void apply_program_chunk(float (&v)[32], const __half* bias, int col0,
                                                    int N, const Epi& epi,
                                                    const EpiProgram& prog) {
#pragma unroll 1
  for (int k = 0; k < epi.n_ops; ++k) {
    const EpiOp op = prog.ops[k];
    switch (op.type) {
      case kOpBias:
        add_bias_chunk(v, bias, col0, N);
        break;
      case kOpRelu:
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = v[i] > 0.0f ? v[i] : 0.0f;
        break;
      case kOpGelu:
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = gelu_erf(v[i]);
        break;
      case kOpScale:
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= op.a;
        break;
      case kOpClamp:
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = fminf(fmaxf(v[i], op.a), op.b);
        break;
      default:  // kOpQuantI8: applied by the store
        break;
    }
  }
}

// Rounds 32 values to FP16 and stores the columns < N of them at drow + col0
// (16-byte stores when `full`: all 32 in range and 16-byte aligned).
__device__ __forceinline__ void store_f16_32(const float (&v)[32], __half* drow, int col0, int N,
                                             bool full) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (full) {
      uint4 ov;
      __half2* oh = reinterpret_cast<__half2*>(&ov);
#pragma unroll
      for (int h = 0; h < 4; ++h) oh[h] = __floats2half2_rn(v[q * 8 + 2 * h], v[q * 8 + 2 * h + 1]);
      *reinterpret_cast<uint4*>(drow + col0 + q * 8) = ov;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (col0 + q * 8 + i < N) drow[col0 + q * 8 + i] = __float2half_rn(v[q * 8 + i]);
    }
  }
}

// int8 codes of 32 values (the program's closing quantization by `scale`),
// stored at qrow + col0 for the columns < N (two 16-byte stores when `full`).
__device__ __forceinline__ void store_i8_32(const float (&v)[32], int8_t* qrow, int col0, int N,
                                           float scale, bool full) {
  if (full) {
    uint32_t w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      w[q] = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b)
        w[q] |= static_cast<uint32_t>(static_cast<uint8_t>(quant_i8(scale * v[q * 4 + b])))
                << (8 * b);
    }
    reinterpret_cast<uint4*>(qrow + col0)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(qrow + col0)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col0 + i < N) qrow[col0 + i] = quant_i8(scale * v[i]);
  }
}

// Fused FP16 epilogue for one thread's row and 32 consecutive columns:
// D = round_fp16(epilogue(alpha*acc + beta*C)), the epilogue being bias then
// GELU (flags) or a program.  C (read only when beta != 0) has leading
// dimension ldc, D has ldd; they are one buffer or do not overlap.  Rows >= M
// and columns >= N are skipped.  16-byte accesses need a 16-byte aligned
// base and a pitch of a multiple of 8 (a batched problem's C and D may start
// anywhere 2-byte aligned); otherwise the chunk takes one element at a time.
__device__ __forceinline__ void epilogue_f16_chunk(const uint32_t (&r)[32], int row, int col0,
                                                   int M, int N, const Epi& epi,
                                                   const EpiProgram& prog, const __half* c,
                                                   int64_t ldc, __half* d, int64_t ldd,
                                                   const __half* bias) {
  if (row >= M) return;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = epi.alpha * __uint_as_float(r[i]);
  __half* drow = d + static_cast<int64_t>(row) * ldd;
  const bool in_range = col0 + 32 <= N;
  const bool full = in_range && ((ldd & 7) == 0) && ((reinterpret_cast<uintptr_t>(d) & 15) == 0);
  if (epi.beta != 0.0f) {
    const __half* crow = c + static_cast<int64_t>(row) * ldc;
    if (in_range && (ldc & 7) == 0 && (reinterpret_cast<uintptr_t>(c) & 15) == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 cv = *reinterpret_cast<const uint4*>(crow + col0 + q * 8);
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
        if (col0 + i < N) v[i] = fmaf(epi.beta, __half2float(crow[col0 + i]), v[i]);
    }
  }
  if (epi.flags & kEpiProgram) {
    apply_program_chunk(v, bias, col0, N, epi, prog);
    if (epi.flags & kEpiOutI8) {  // D is int8: ldd counts bytes
      int8_t* qrow = reinterpret_cast<int8_t*>(d) + static_cast<int64_t>(row) * ldd;
      const bool full8 = in_range && ((ldd & 15) == 0) &&
                         ((reinterpret_cast<uintptr_t>(d) & 15) == 0);
      store_i8_32(v, qrow, col0, N, prog.ops[epi.n_ops - 1].a, full8);
      return;
    }
    store_f16_32(v, drow, col0, N, full);
    return;
  }
  if (epi.flags & kEpiBias) add_bias_chunk(v, bias, col0, N);
  const bool gelu = (epi.flags & kEpiGelu) != 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {  // 8 values at a time: activation, rounding, store
    if (gelu) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[q * 8 + i] = gelu_erf(v[q * 8 + i]);
    }
    if (full) {
      uint4 ov;
      __half2* oh = reinterpret_cast<__half2*>(&ov);
#pragma unroll
      for (int h = 0; h < 4; ++h) oh[h] = __floats2half2_rn(v[q * 8 + 2 * h], v[q * 8 + 2 * h + 1]);
      *reinterpret_cast<uint4*>(drow + col0 + q * 8) = ov;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (col0 + q * 8 + i < N) drow[col0 + q * 8 + i] = __float2half_rn(v[q * 8 + i]);
    }
  }
}

// ------------------------------------------------------ staged (TMA) epilogue
// A warp's 32 accumulator rows x 32 columns pass through a shared-memory box
// that TMA fills with C and drains to D in whole lines, instead of each
// thread touching 32 different rows of global memory per access.  The box is
// 32 rows of 64 bytes in the 64-byte swizzle of the C/D tensor map: the
// 16-byte piece q of row r sits at r*64 + ((q ^ ((r >> 1) & 3)) * 16).
// Thread r of the warp touches row r only, and any 8 consecutive rows cover
// all 32 banks, so its 16-byte accesses are free of bank conflicts.
constexpr int kEpiBoxRows = 32;
constexpr int kEpiBoxCols = 32;
constexpr int kEpiBoxBytes = kEpiBoxRows * kEpiBoxCols * 2;

__device__ __forceinline__ uint32_t epi_box_offset(int r, int q) {
  return static_cast<uint32_t>(r * 64 + ((q ^ ((r >> 1) & 3)) << 4));
}

// D = round_fp16(epilogue(alpha*acc + beta*C)) for row `r` of a staged
// box whose first column is D column col0; with `has_c` the box holds C on
// entry.  D replaces C in the box.  Columns >= N (bias only) read 0; the
// store's tensor map drops them.
__device__ __forceinline__ void epilogue_f16_box(const uint32_t (&acc)[32], uint8_t* box, int r,
                                                 int col0, int N, const Epi& epi,
                                                 const EpiProgram& prog, const __half* bias,
                                                 bool has_c) {
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = epi.alpha * __uint_as_float(acc[i]);
  if (has_c) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 cv = *reinterpret_cast<const uint4*>(box + epi_box_offset(r, q));
      const __half2* ch = reinterpret_cast<const __half2*>(&cv);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float2 f = __half22float2(ch[h]);
        v[q * 8 + 2 * h] = fmaf(epi.beta, f.x, v[q * 8 + 2 * h]);
        v[q * 8 + 2 * h + 1] = fmaf(epi.beta, f.y, v[q * 8 + 2 * h + 1]);
      }
    }
  }
  const bool program = (epi.flags & kEpiProgram) != 0;
  if (program)
    apply_program_chunk(v, bias, col0, N, epi, prog);
  else if (epi.flags & kEpiBias)
    add_bias_chunk(v, bias, col0, N);
  const bool gelu = !program && (epi.flags & kEpiGelu) != 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {  // 8 values at a time: activation, rounding, staging
    if (gelu) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[q * 8 + i] = gelu_erf(v[q * 8 + i]);
    }
    uint4 ov;
    __half2* oh = reinterpret_cast<__half2*>(&ov);
#pragma unroll
    for (int h = 0; h < 4; ++h) oh[h] = __floats2half2_rn(v[q * 8 + 2 * h], v[q * 8 + 2 * h + 1]);
    *reinterpret_cast<uint4*>(box + epi_box_offset(r, q)) = ov;
  }
}

// ------------------------------------------------- exact INT32 from FP32 chunks
// An INT8 x INT8 product is an integer of magnitude <= 2^14, so a sum of at
// most 1024 of them is an integer of magnitude <= 2^24, exact in FP32.  The
// integer kernels accumulate K in chunks of this many 64-wide K blocks and
// carry an INT32 running sum between chunks.
constexpr int kI32ChunkKb = 16;  // 16 x 64 = 1024

__device__ __forceinline__ void tmem_st_32cols(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tc_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// C and D of an INT32 output: C read when beta != 0, leading dimensions in
// elements; the two are one buffer or do not overlap.
struct I32Out {
  const int32_t* c;
  int64_t ldc;
  int32_t* d;
  int64_t ldd;
};

// INT32 output of one 32-column chunk: D = alpha*sum + beta*C (mod 2^32).
__device__ __forceinline__ void store_i32_chunk(const uint32_t (&s)[32], int row, int col0, int M,
                                                int N, int32_t alpha, int32_t beta,
                                                const I32Out& o) {
  if (row >= M) return;
  const int32_t* crow = o.c + static_cast<int64_t>(row) * o.ldc;
  int32_t* drow = o.d + static_cast<int64_t>(row) * o.ldd;
  const uint32_t al = static_cast<uint32_t>(alpha), be = static_cast<uint32_t>(beta);
  const bool full = (col0 + 32 <= N) && (((o.ldc | o.ldd) & 3) == 0) &&
                    (((reinterpret_cast<uintptr_t>(o.c) | reinterpret_cast<uintptr_t>(o.d)) & 15) == 0);
  if (full) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint4 v;
      if (be != 0u) v = *reinterpret_cast<const uint4*>(crow + col0 + q * 4);
      else v = make_uint4(0, 0, 0, 0);
      v.x = al * s[q * 4 + 0] + be * v.x;
      v.y = al * s[q * 4 + 1] + be * v.y;
      v.z = al * s[q * 4 + 2] + be * v.z;
      v.w = al * s[q * 4 + 3] + be * v.w;
      *reinterpret_cast<uint4*>(drow + col0 + q * 4) = v;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (col0 + i < N) {
        const uint32_t c = be != 0u ? static_cast<uint32_t>(crow[col0 + i]) : 0u;
        drow[col0 + i] = static_cast<int32_t>(al * s[i] + be * c);
      }
    }
  }
}

// One 32-column piece of an INT8 accumulation chunk: convert the exact FP32
// chunk sums `r` to INT32, add the running sum kept in TMEM at `sums` (all
// chunks but the first), then either store the new running sum back (not the
// last chunk) or write the result to D (last chunk).
__device__ __forceinline__ void flush_i32_piece(uint32_t (&r)[32], uint32_t sums, bool first,
                                                bool last, int row, int col0, int M, int N,
                                                int32_t alpha, int32_t beta, const I32Out& o) {
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = static_cast<uint32_t>(__float2int_rn(__uint_as_float(r[i])));
  if (!first) {
    uint32_t s[32];
    tmem_ld_32cols(sums, s);
    tc_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] += s[i];
  }
  if (!last) {
    tmem_st_32cols(sums, r);
    tc_wait_st();
  } else if (col0 < N) {
    store_i32_chunk(r, row, col0, M, N, alpha, beta, o);
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
  constexpr int kCache = 64;
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

// C or D of the staged epilogue: M x N FP16, row pitch ld elements, boxes
// of 32 x 32 in the 64-byte swizzle.  Needs ld % 8 == 0 and a 16-byte
// aligned base.
inline cudaError_t make_f16_epi_map(CUtensorMap* map, const void* base, int64_t M, int64_t N,
                                    int64_t ld) {
  return make_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, M, N, ld * 2, kEpiBoxRows,
                     kEpiBoxCols, CU_TENSOR_MAP_SWIZZLE_64B);
}

// D of the INT32 output: M x N INT32, row pitch ld elements, boxes of 32
// rows x 16 columns (64-byte rows, the same 64-byte swizzle).  Needs
// ld % 4 == 0 and a 16-byte aligned base.
inline cudaError_t make_i32_epi_map(CUtensorMap* map, const void* base, int64_t M, int64_t N,
                                    int64_t ld) {
  return make_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_INT32, base, M, N, ld * 4, kEpiBoxRows,
                     kEpiBoxCols / 2, CU_TENSOR_MAP_SWIZZLE_64B);
}

// K-major FP16 operand tile: box_rows x 64 elements, 128-byte swizzle.
inline cudaError_t make_f16_kmajor_map(CUtensorMap* map, const void* base, int64_t rows, int64_t k,
                                       int64_t ld, int box_rows) {
  return make_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, rows, k, ld * 2, box_rows,
                     kBlockK, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace tc
}  // namespace dg
