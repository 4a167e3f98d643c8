/*
 * dg.h -- C ABI of libdg, a GEMM library for one NVIDIA GB300 GPU (sm_103a).
 *
 *   D = epilogue(alpha * A.B + beta * C)
 *
 * The operation is the one stated in the "DeepGEMM" articles this library
 * follows (kwkr.cn/news/562171, section 3.2 step 3: the fused epilogue
 * "alpha * C + beta * D" and the launch argument order A, B, C, alpha, beta,
 * m, n, k; section 2.2 third layer: bias and GELU fused into the GEMM;
 * discosf.com/news/5532976, section 2.2 layer 2: the precision triple
 * {weight, activation, output}, e.g. int4_e2m1 x fp16 -> fp16; section 3.5:
 * FP32 accumulation with an FP16 output cast).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All sizes are element counts of type int64_t.
 *  - A is M x K, row-major, leading dimension lda (elements, lda >= K).
 *  - B is K x N stored "column-major": N rows of K contiguous elements,
 *    leading dimension ldb (elements, ldb >= K).  For DG_E2M1, B holds two
 *    4-bit codes per byte: byte p of a row carries k = 2p in its low nibble
 *    and k = 2p+1 in its high nibble; ldb counts codes, is even, and a row is
 *    ldb/2 bytes long.
 *  - C (input, read only when beta != 0) and D (output) share one buffer,
 *    row-major M x N with leading dimension N (BLAS in/out convention).  Its
 *    type is FP16 for the floating-point pairs and INT32 for INT8 x INT8.
 *  - bias is FP16 [N], read only by the bias epilogues.
 *  - Every pointer is caller-owned device memory; libdg never frees it.
 *  - A and B must be 16-byte aligned and lda/ldb must span a multiple of 16
 *    bytes (the tensor-memory-access engine reads them in tiles); C must be
 *    16-byte aligned; bias 2-byte aligned.
 *  - Any host thread may call.  The library's own state (device
 *    descriptors, cached plans, scratch buffers kept per device and stream,
 *    one-time kernel set-up) is guarded internally, so calls on different
 *    streams from different threads are independent.  Calls on one stream
 *    must not overlap on the host: a call may grow that stream's scratch
 *    and free the buffer another call is about to launch with.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *    Invalid arguments are rejected synchronously, before any launch, with a
 *    status and a message in dg_last_error().  Faults in a launched kernel
 *    surface at the caller's next synchronisation (CUDA semantics); a kernel
 *    whose internal pipeline wait runs past its time limit records
 *    DG_ERR_TIMEOUT in a per-device status word that dg_check_status() reads.
 */
#ifndef DG_H_
#define DG_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the runtime type is a pointer to this opaque struct). */
typedef struct CUstream_st *dg_stream_t;

typedef enum {
  DG_OK = 0,
  DG_ERR_INVALID_ARG = 1,        /* null/misaligned pointer, bad size or leading dimension */
  DG_ERR_UNSUPPORTED = 2,        /* dtype pair, epilogue or scalar this path does not take */
  DG_ERR_NO_VALID_CANDIDATE = 3, /* the planner found no tile that meets every constraint */
  DG_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed */
  DG_ERR_TIMEOUT = 5,            /* a device-side pipeline wait ran past its limit */
  DG_ERR_INVALID_STATE = 6       /* no usable device, or a plan that does not fit the call */
} dg_status;

/* Input element types (the output type follows from the pair). */
typedef enum {
  DG_F16 = 0,   /* IEEE binary16 */
  DG_I8 = 1,    /* two's-complement int8 */
  DG_E2M1 = 2,  /* 4-bit float: sign | 2-bit exponent (bias 1) | 1-bit mantissa */
  DG_MXF4 = 3   /* block-scaled E2M1 (MXFP4): E2M1 codes packed as for DG_E2M1, plus one
                   E8M0 scale byte (2^(e - 127); 255 = NaN) per 32 codes along K.  Taken by
                   dg_quantize_mxf4, dg_gemm_mxf4 and dg_plan_tiles (pair DG_MXF4 x DG_MXF4) */
} dg_dtype;

/* Fused epilogue applied to t = alpha*acc + beta*C:  bias adds bias[j] to t,
 * GELU takes 0.5*t*(1 + erf(t/sqrt(2))) (after the bias when both are set). */
typedef enum {
  DG_EPI_NONE = 0,
  DG_EPI_BIAS = 1,
  DG_EPI_GELU = 2,
  DG_EPI_BIAS_GELU = 3
} dg_epilogue;

/* Epilogue programs: the op_type registry of the pages' epilogue generator
 * (kwkr.cn/news/562171, section 2.2 third layer: post-processing such as
 * bias add, ReLU and quantization fused into the GEMM; discosf.com/news/
 * 5532976, section 6.1: an epilogue chosen by op_type, e.g. "gelu").  A
 * program is up to DG_MAX_EPILOGUE_OPS ops applied in order to
 * t = alpha*acc + beta*C, in FP32, before the single rounding to FP16. */
#define DG_MAX_EPILOGUE_OPS 8
typedef enum {
  DG_OP_BIAS = 1,  /* t += bias[j] (FP16 [N]) */
  DG_OP_RELU = 2,  /* t = max(t, 0); a NaN t becomes 0 */
  DG_OP_GELU = 3,  /* t = 0.5*t*(1 + erf(t/sqrt(2))) */
  DG_OP_SCALE = 4, /* t = t * a (e.g. a dequantization or output scale) */
  DG_OP_CLAMP = 5, /* t = min(max(t, a), b), a <= b (saturation before a narrow output);
                      a NaN t becomes a */
  DG_OP_QUANT_I8 = 6 /* last op only: D is int8, D = round-half-to-even(a * t) saturated to
                        [-128, 127], a NaN to 0 (output quantization); ldd counts bytes */
} dg_op_type;

typedef struct {
  int type;    /* dg_op_type */
  float a, b;  /* operands of DG_OP_SCALE (a) and DG_OP_CLAMP (a, b); ignored otherwise */
} dg_epilogue_op;

typedef struct {
  int n_ops; /* 0 .. DG_MAX_EPILOGUE_OPS */
  dg_epilogue_op ops[DG_MAX_EPILOGUE_OPS];
} dg_epilogue_program;

/* Kernel families a plan can select. */
typedef enum {
  DG_KERNEL_TC = 0,    /* tensor-core pipeline: TMA -> SMEM ring -> tcgen05.mma -> TMEM -> fused
                          epilogue (MXFP4: packed codes on the block-scaled kind::mxf4 MMA) */
  DG_KERNEL_GEMV = 1,  /* thin-M split-K streaming kernel on the CUDA cores */
  DG_KERNEL_TC_WIDENED = 2, /* int8 / E2M1 operands widened to FP16 by a streaming pre-pass into
                               a library workspace, then the FP16 tensor-core kernel (INT8:
                               exact INT32 output) -- for compute-bound shapes; MXFP4
                               operands are widened to BF16 with their block scales */
  DG_KERNEL_SKINNY = 3, /* FP16 x E2M1 with M <= 16 (HBM-bound): packed weights streamed into
                           registers, widened there and fed to warp-level m16n8k16 MMAs */
  DG_KERNEL_GEMV_MMA = 4, /* FP16 x FP16 with 2 <= M <= 16 (HBM-bound): the split-K GEMV's
                            streaming of B rows, multiplied on warp-level m16n8k16 MMAs */
  DG_KERNEL_TC_STREAMK = 5 /* FP16 x FP16 tensor-core pipeline with stream-K work division
                              (kwkr.cn/news/562171, section 2.2 first layer: the K step of
                              each piece of work chosen so that ragged tile counts fill every
                              SM): the tiles that fill whole waves run whole, the K blocks of
                              the rest are cut into one even range per CTA (pair); a tile
                              split between ranges is finished by the range holding its first
                              K block, which adds the others' FP32 partials in a fixed order
                              (results are bit-stable run to run).  Partials and flags live
                              in a library workspace per device and stream.  D and C (when
                              beta != 0) need 16-byte aligned bases and rows (ldd, ldc
                              multiples of 8) and no int8 output; other layouts, and shapes
                              whose tiles fill whole waves, run the data-parallel kernel of
                              the same tile.  The plan's grid is the CTAs the work is divided
                              over (those left without work are not launched) and split_k the
                              most ranges one tile meets */
} dg_kernel;

/* Hardware description the planner solves against
 * (kwkr.cn/news/562171, section 3.2 step 1: compute capability, shared memory
 * per SM, L2 size, threads per SM, tensor-core types; extended here with the
 * resources a Blackwell SM exposes). */
typedef struct {
  int sm_count;
  int cc_major, cc_minor;
  int smem_per_block_optin;   /* bytes one CTA may use */
  int smem_per_sm;            /* bytes per SM */
  int regs_per_sm;            /* 32-bit registers per SM */
  int regs_per_thread_max;
  int max_threads_per_sm;
  int tmem_cols;              /* tensor-memory columns per SM (128 lanes x 32 bit each); 0 = none */
  int64_t l2_bytes;
  double hbm_gbps;            /* bytes/ns; 0 = unknown */
  double tc_f16_tflops;       /* dense FP16 tensor rate; 0 = unknown */
  double clock_ghz;
} dg_hw_desc;

/* One tile plan (kwkr.cn/news/562171, section 2.2 first layer: a solution
 * (M_tile, N_tile, K_tile) of the shared-memory / register / occupancy
 * constraint system; here with split-K, pipeline depth and CTA pairing). */
typedef struct {
  int kernel;       /* dg_kernel */
  int m_tile;       /* rows of D per CTA (or per CTA pair when cta_group == 2) */
  int n_tile;       /* columns of D per CTA */
  int k_tile;       /* K elements per pipeline stage */
  int split_k;      /* number of K slices reduced deterministically (1 = none) */
  int stages;       /* shared-memory ring depth */
  int cta_group;    /* 1, or 2 for a tcgen05 CTA pair */
  int swap_ab;      /* 1: the kernel computes D^T = B^T.A^T (thin-M tensor path) */
  int smem_bytes;   /* dynamic shared memory of the launch */
  int threads;      /* threads per CTA */
  int regs_per_thread; /* registers per thread the register constraint was checked with: the
                          kernel's own figure (cudaFuncGetAttributes) when a device is present,
                          else the planner's upper bound for that kernel */
  int grid;         /* CTAs launched */
  double occupancy; /* wave efficiency: work units / (waves * SMs) */
  double est_us;    /* cost-model time */
  double est_tflops;
} dg_tile_plan;

/* Fill *out for CUDA device `device` from cudaDeviceGetAttribute.
 * Returns DG_ERR_INVALID_STATE when no such device exists. */
dg_status dg_query_hw(int device, dg_hw_desc *out);

/* The tile planner (kwkr.cn/news/562171, section 2.2 first layer and
 * section 3.2 step 2; discosf.com/news/5532976, section 4.1 stage 2).
 * Enumerates the tile space of the kernels this library ships, keeps the
 * candidates whose shared memory, tensor memory, registers and threads fit
 * `hw` and whose wave efficiency is at least target_occupancy, and writes up
 * to max_out of them to out[], best estimated time first.  *n_out receives
 * the number written.  hw == NULL means the current device.  Host only: no
 * GPU work.  DG_ERR_NO_VALID_CANDIDATE when nothing survives the pruning. */
dg_status dg_plan_tiles(int64_t M, int64_t N, int64_t K, dg_dtype dtype_a, dg_dtype dtype_b,
                        dg_epilogue epilogue, const dg_hw_desc *hw, double target_occupancy,
                        dg_tile_plan *out, int max_out, int *n_out);

/* D = epilogue(alpha * A.B + beta * C) with the planner's best plan.
 * Supported pairs: F16 x F16 and F16 x E2M1 (FP32 accumulation, FP16 out,
 * any epilogue) and I8 x I8 (exact INT32 accumulation, INT32 out, no
 * epilogue, integral alpha and beta, wrap-around modulo 2^32).
 * M == 0 or N == 0 is a no-op; K == 0 gives epilogue(beta * C).
 * May grow a per-(device, stream) split-K workspace the first time a shape
 * needs it (cudaMalloc; libdg owns it until dg_shutdown).  Under CUDA-graph
 * capture, make one call of the same shape on the capturing stream before
 * capture begins (or use dg_gemm_thin_noalloc), so no allocation happens
 * while capturing. */
dg_status dg_gemm(int64_t M, int64_t N, int64_t K, dg_dtype dtype_a, dg_dtype dtype_b,
                  const void *A, int64_t lda, const void *B, int64_t ldb, void *C,
                  const void *bias, float alpha, float beta, dg_epilogue epilogue,
                  dg_stream_t stream);

/* D = epilogue(alpha * A.B + beta * C) on HOST buffers: the same operation
 * and rules as dg_gemm, with the host-to-device and device-to-host copies
 * inside the call.  This is the pages' calling pattern (discosf.com/news/
 * 5532976, section 3.4: page-locked host matrices are bound to the GEMM, and
 * the runtime allocates device memory on demand at the first launch and
 * manages its lifetime; no cudaMalloc or cudaMemcpy in the caller).
 *   A, B, bias: host inputs in dg_gemm's layouts (A: M rows of lda elements,
 *     B: N rows of ldb elements / codes, bias: N FP16); C: host input (M x N,
 *     leading dimension N; FP16, or INT32 for I8 x I8), read only when
 *     beta != 0 and may then be NULL otherwise; D: host output of the same
 *     layout as C (may equal C).
 *   Copies and kernels are asynchronous and ordered on `stream`: the caller
 *   synchronises that stream before reading D or reusing the inputs.  With
 *   page-locked (pinned) host memory the copies overlap one another and the
 *   kernels: B and bias are copied first, then row panels of A and C are
 *   copied, multiplied and copied back on two internal streams joined back to
 *   `stream`.  Pageable memory works, with copies that do not overlap.
 *   Device copies of the operands live in a per-(device, stream) workspace
 *   that grows with cudaMalloc and that libdg owns until dg_shutdown.
 * Errors: as dg_gemm, plus DG_ERR_INVALID_ARG for a NULL D, or a NULL C with
 * beta != 0, and DG_ERR_CUDA for a failed copy. */
dg_status dg_gemm_host(int64_t M, int64_t N, int64_t K, dg_dtype dtype_a, dg_dtype dtype_b,
                       const void *A, int64_t lda, const void *B, int64_t ldb, const void *C,
                       void *D, const void *bias, float alpha, float beta,
                       dg_epilogue epilogue, dg_stream_t stream);

/* D = program(alpha * A.B + beta * C) with separate C and D buffers.
 * The general form of dg_gemm (kwkr.cn/news/562171, section 3.2 step 3: the
 * generated kernel takes A, B, C, alpha, beta; section 2.2 third layer: the
 * fused post-processing ops), BLAS-style: C is read, D is written.
 *   C: M x N, leading dimension ldc >= N, read only when beta != 0 (may then
 *     be NULL otherwise); D: M x N, leading dimension ldd >= N.  Both FP16,
 *     or INT32 for I8 x I8; both 16-byte aligned.  C and D are the same
 *     buffer with ldc == ldd (in place) or do not overlap; columns N .. ld-1
 *     of D are never written.
 *   program: NULL or n_ops == 0 for none.  For I8 x I8 (exact INT32 output)
 *     it must be empty.  DG_OP_BIAS needs bias (FP16 [N]), which is read
 *     only by that op.  A program ending in DG_OP_QUANT_I8 makes D int8 (C,
 *     when read, stays FP16), so C and D must then be different buffers.
 *   Plan, kernels, workspaces and errors as dg_gemm; DG_ERR_INVALID_ARG for
 *   ldc < N (with beta != 0), ldd < N, a NULL D, more than
 *   DG_MAX_EPILOGUE_OPS ops, an unknown op type, a clamp with a > b (or a
 *   NaN bound), a non-finite scale, DG_OP_QUANT_I8 before the last op, or an
 *   int8 D that is also C; DG_ERR_UNSUPPORTED for a program on I8 x I8. */
dg_status dg_gemm_ex(int64_t M, int64_t N, int64_t K, dg_dtype dtype_a, dg_dtype dtype_b,
                     const void *A, int64_t lda, const void *B, int64_t ldb, const void *C,
                     int64_t ldc, void *D, int64_t ldd, const void *bias, float alpha, float beta,
                     const dg_epilogue_program *program, dg_stream_t stream);

/* A strided batch of independent problems of one shape:
 *   D_z = epilogue(alpha * A_z.B_z + beta * C_z),  z = 0 .. batch-1,
 * with A_z = A + z*stride_a, B_z = B + z*stride_b, C_z (= D_z) = C + z*stride_c
 * and bias_z = bias + z*stride_bias.  For the pages' many small GEMMs of one
 * shape, e.g. the attention QKV projections M=1, N=128, K=4096
 * (discosf.com/news/5532976, section 5.3, third stage).
 *   Strides are element counts (codes for E2M1 B), >= 0; 0 shares the
 *   operand between problems (e.g. one bias for all).  With batch > 1,
 *   stride_c >= M*N (outputs may not overlap) and stride_a and stride_b span
 *   multiples of 16 bytes, so every problem's A and B keep dg_gemm's
 *   alignment; stride_c may be any such count (C and D of problem z > 0 need
 *   only their element alignment).  Each problem otherwise follows dg_gemm's
 *   layouts and rules.
 *   When the planner picks the thin split-K GEMV for the shape (FP16, M <= 8)
 *   the whole batch is one launch; otherwise each problem is launched in
 *   turn on `stream`.  The GEMV's split-K workspace grows with the batch.
 *   batch == 0 is a no-op.
 * Errors: as dg_gemm, plus DG_ERR_INVALID_ARG for a negative batch or
 * stride, overlapping outputs or a misaligned stride_a / stride_b. */
dg_status dg_gemm_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K,
                                  dg_dtype dtype_a, dg_dtype dtype_b, const void *A, int64_t lda,
                                  int64_t stride_a, const void *B, int64_t ldb, int64_t stride_b,
                                  void *C, int64_t stride_c, const void *bias,
                                  int64_t stride_bias, float alpha, float beta,
                                  dg_epilogue epilogue, dg_stream_t stream);

/* A group of independent problems that share N, K, the dtypes, scalars and
 * epilogue but not M or their buffers, e.g. the experts of a mixture-of-
 * experts layer, each with the rows routed to it (a grouped form of the many
 * small GEMMs of discosf.com/news/5532976, section 5.3, third stage):
 *   D_g = epilogue(alpha * A_g.B_g + beta * C_g),  g = 0 .. count-1.
 *   Ms, A, B, C and bias are HOST arrays of count entries: row counts (0
 *   skips the problem) and device pointers in dg_gemm's layouts (lda, ldb
 *   shared; C_g / D_g leading dimension N).  bias may be NULL without a bias
 *   epilogue; entries of a problem with M = 0 are not read.
 *   FP16 x FP16 groups whose largest M is at most 16 run as ONE launch of the
 *   warp-MMA GEMV: a table of the problems is copied (cudaMemcpyAsync from
 *   pageable memory, so not under CUDA-graph capture) to a per-(device,
 *   stream) workspace, with the split-K workspace sized for the group.  Other
 *   groups launch each problem in turn on `stream`.
 * Errors: as dg_gemm for each problem (the message names the problem), plus
 * DG_ERR_INVALID_ARG for a negative count or M or a NULL array. */
dg_status dg_gemm_grouped(int64_t count, const int64_t *Ms, int64_t N, int64_t K,
                          dg_dtype dtype_a, dg_dtype dtype_b, const void *const *A, int64_t lda,
                          const void *const *B, int64_t ldb, void *const *C,
                          const void *const *bias, float alpha, float beta,
                          dg_epilogue epilogue, dg_stream_t stream);

/* Block quantization of an FP16 matrix to MXFP4, row by row along K: for
 * each block of 32 values (the last block of a row holds K mod 32 when K is
 * not a multiple of 32) the scale is X = 2^s with s = floor(log2(amax)) - 2
 * (amax the block's largest magnitude; an all-zero block takes s = -127),
 * stored as the E8M0 byte s + 127, and each value becomes the E2M1 code
 * nearest to v / X (ties to the code with mantissa bit 0, magnitudes above 6
 * saturated to 6, the sign kept, so a negative value that rounds to 0 gives
 * code 8).  A block holding a NaN or an infinity gets the scale byte 255 and
 * codes 0.  The pages ask for low-bit operands in the tensor cores' own
 * formats (discosf.com/news/5532976, section 2.2 layer 2 and section 4.3)
 * without fixing a block format; this is the MX block format those
 * tensor cores' block-scaled MMAs consume.
 *   X: rows x K FP16, leading dimension ldx >= K elements, ldx * 2 a multiple
 *     of 16 bytes, X 16-byte aligned.
 *   codes: rows x K codes packed two per byte (byte p of a row: k = 2p in the
 *     low nibble, k = 2p + 1 in the high nibble), leading dimension ldq
 *     codes: ldq >= K and a multiple of 32 (16-byte rows), 16-byte aligned.
 *     Bytes of a row past ceil(K / 2) are not written; with K odd, the high
 *     nibble of the last byte is written as 0.
 *   scales: rows x ceil(K / 32) bytes, leading dimension lds >= ceil(K / 32)
 *     bytes; bytes past ceil(K / 32) are not written.
 *   One launch on `stream`; rows == 0 or K == 0 is a no-op.  Every pointer is
 *   caller-owned device memory.
 * Errors: DG_ERR_INVALID_ARG for negative sizes, NULL or misaligned pointers
 * and leading dimensions that break the rules above. */
dg_status dg_quantize_mxf4(int64_t rows, int64_t K, const void *X, int64_t ldx, void *codes,
                           int64_t ldq, void *scales, int64_t lds, dg_stream_t stream);

/* D = epilogue(alpha * A.B + beta * C) for MXFP4 operands: A (M x K) and B
 * (N rows of K), each as packed E2M1 codes (layout of dg_quantize_mxf4's
 * output; lda, ldb in codes, >= K and multiples of 32) plus E8M0 scale bytes
 * (scale_a: M rows of lds_a >= ceil(K / 32) bytes; scale_b: N rows of
 * lds_b bytes).  Element k of a row stands for e2m1(code) * 2^(e - 127), with
 * e the scale byte of block k / 32 (255: NaN for the whole block).
 * Products are summed in FP32; C, D (one buffer, M x N, leading dimension N,
 * FP16), bias, the epilogue, alpha and beta are as in dg_gemm.
 * Runs the plan dg_plan_tiles gives for the pair DG_MXF4 x DG_MXF4:
 *  - DG_KERNEL_TC (K even): the codes go to the tensor cores as stored, on
 *    block-scaled kind::mxf4 MMAs with FP32 accumulation; the kernel reads
 *    the scale bytes where they are when each operand's scale rows start on
 *    16-byte boundaries (pointer and lds multiples of 16), and otherwise
 *    first copies them to a 16-byte pitch in a per-(device, stream)
 *    workspace (M or N times ceil(K / 32) rounded up to 16 bytes).  Codes
 *    past K (and, for the scales, blocks past ceil(K / 32)) are never read.
 *  - DG_KERNEL_TC_WIDENED (any K; the only plan for odd K): both operands
 *    are widened with their scales into a BF16 copy in that workspace (exact:
 *    each value has at most two significant bits and BF16 keeps FP32's
 *    exponent range; scale bytes above 251 may overflow to an infinity),
 *    then kind::f16 MMAs multiply the copies.
 * M == 0 or N == 0 is a no-op; K == 0 gives epilogue(beta * C).
 * The workspace grows with cudaMalloc the first time a shape needs it:
 * under CUDA-graph capture, make one call of the same shape on the
 * capturing stream before capture begins.
 * Errors: as dg_gemm, plus DG_ERR_INVALID_ARG for NULL or misaligned scale
 * pointers and leading dimensions that break the rules above. */
dg_status dg_gemm_mxf4(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                       const void *scale_a, int64_t lds_a, const void *B, int64_t ldb,
                       const void *scale_b, int64_t lds_b, void *C, const void *bias, float alpha,
                       float beta, dg_epilogue epilogue, dg_stream_t stream);

/* As dg_gemm_mxf4, but runs `plan` (one returned by dg_plan_tiles for the
 * same M, N, K and the pair DG_MXF4 x DG_MXF4): DG_KERNEL_TC is the
 * block-scaled MMA on the packed codes, DG_KERNEL_TC_WIDENED the BF16
 * widening.  The pages' planner hands its chosen tile to the generated
 * kernel the same way (kwkr.cn/news/562171, section 3.2 steps 2 and 4).
 * DG_ERR_INVALID_STATE when the plan does not fit (e.g. a DG_KERNEL_TC plan
 * with an odd K); DG_ERR_INVALID_ARG for a NULL plan; otherwise as
 * dg_gemm_mxf4. */
dg_status dg_gemm_mxf4_planned(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                               const void *scale_a, int64_t lds_a, const void *B, int64_t ldb,
                               const void *scale_b, int64_t lds_b, void *C, const void *bias,
                               float alpha, float beta, dg_epilogue epilogue,
                               const dg_tile_plan *plan, dg_stream_t stream);

/* As dg_gemm, but runs `plan` (one returned by dg_plan_tiles for the same
 * M, N, K and dtypes).  DG_ERR_INVALID_STATE when the plan does not fit. */
dg_status dg_gemm_planned(int64_t M, int64_t N, int64_t K, dg_dtype dtype_a, dg_dtype dtype_b,
                          const void *A, int64_t lda, const void *B, int64_t ldb, void *C,
                          const void *bias, float alpha, float beta, dg_epilogue epilogue,
                          const dg_tile_plan *plan, dg_stream_t stream);

/* Thin-M GEMM that allocates nothing.  The pages have no counterpart: this
 * entry point exists for callers that cannot let a library call cudaMalloc
 * (code that runs while a CUDA graph is being captured, runtimes that own all
 * device memory through their own pool, locked-down allocators).
 * Computes the same GEMM as dg_gemm, for F16 x F16 with M <= 8, within the
 * same error bound, but always through the split-K GEMV kernel on the CUDA
 * cores with that kernel's own best split.  dg_gemm may choose another
 * kernel (the warp-MMA GEMV or a tensor-core plan for 2 <= M <= 8) or another
 * split for the same shape, so the two agree within the bound, not bit for
 * bit.  The FP32 partial sums and arrival counters live in a file-scope
 * static device array of 2 MiB + 64 KiB that every GPU loading the library
 * holds until exit.
 *  - The first call on a device looks the array's device address up with
 *    cudaGetSymbolAddress and reads the device's attributes (once per
 *    device, that device current); make that first call before any stream
 *    capture.
 *  - Shapes whose split-K partials (split * M * N * 4 bytes) or counters
 *    (ceil(N/8) * 4 bytes) exceed the array are rejected with
 *    DG_ERR_INVALID_ARG and a message (a guard: the GEMV's split choice
 *    stays far below both limits for every M <= 8); other pairs or M > 8
 *    give DG_ERR_UNSUPPORTED.
 *  - Every call shares the one array and it keeps the last call's contents:
 *    the call clears the counters on `stream` first (cudaMemsetAsync), and
 *    calls that overlap on the GPU (other streams, other host threads) race.
 *  - Calls no cudaMalloc/cudaFree and no allocating routine.  Arguments,
 *    layouts and errors otherwise as dg_gemm. */
dg_status dg_gemm_thin_noalloc(int64_t M, int64_t N, int64_t K, dg_dtype dtype_a,
                               dg_dtype dtype_b, const void *A, int64_t lda, const void *B,
                               int64_t ldb, void *C, const void *bias, float alpha, float beta,
                               dg_epilogue epilogue, dg_stream_t stream);

/* Message for the last failing call on this thread ("" if none).  Valid
 * until the next libdg call on the same thread. */
const char *dg_last_error(void);

/* Synchronises `stream`, then reads and clears the current device's status
 * word: DG_ERR_TIMEOUT if a kernel gave up on a pipeline wait since the last
 * check, DG_ERR_CUDA if the stream reports an error, else DG_OK. */
dg_status dg_check_status(dg_stream_t stream);

/* Time limit of every device-side pipeline wait, in nanoseconds
 * (default 1e9).  0 restores the default.  Applies to later launches. */
dg_status dg_set_wait_timeout_ns(uint64_t ns);

/* Test hook: one CTA waits on a barrier that nothing completes, with the
 * current time limit, then records DG_ERR_TIMEOUT in the status word and
 * returns.  Lets a test exercise the timeout path without a fault. */
dg_status dg_selftest_wait_timeout(dg_stream_t stream);

/* Kernels launched by this process through libdg so far. */
uint64_t dg_launch_count(void);

/* Frees what libdg allocated on every device (split-K, widened-operand,
 * group-table and host-call workspaces, internal streams and events, status
 * words) and forgets the cached plans; the next call sets them up again.
 * Not to be called while another thread is inside libdg or while its kernels
 * may still run.  Each kernel's shared-memory opt-in is made once per device
 * and process and is not undone: a process that resets a device
 * (cudaDeviceReset) cannot use libdg on that device afterwards. */
dg_status dg_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* DG_H_ */
