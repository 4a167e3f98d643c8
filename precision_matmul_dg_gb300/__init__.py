"""Python binding of libdg (ctypes): argument marshalling only.

Every step of the GEMM runs in libdg's CUDA kernels.  This module loads the
in-tree ``libdg.so`` (built by ``precision_matmul_dg_gb300.build``), declares
the C signatures of ``include/dg.h`` and turns tensors into pointers and
leading dimensions.  PyTorch is used for device memory and streams only.
There is no fallback: if the library is missing, every call raises.
"""

import ctypes
import os

__all__ = [
    "DgError", "F16", "I8", "E2M1", "EPILOGUES", "lib", "lib_path", "gemm", "gemm_raw",
    "gemm_host", "gemm_host_raw", "gemm_ex", "gemm_ex_raw", "gemm_batched", "gemm_grouped",
    "gemm_strided_batched_raw", "prepare_grouped", "OPS", "MAX_EPILOGUE_OPS", "MXF4", "quantize_mxf4",
    "quantize_mxf4_raw", "gemm_mxf4", "gemm_mxf4_raw",
    "EpilogueOp", "EpilogueProgram", "make_program",
    "plan_tiles", "query_hw", "last_error", "check_status", "set_wait_timeout_ns",
    "selftest_wait_timeout", "launch_count", "shutdown", "HwDesc", "TilePlan", "EXPORTS",
]

F16, I8, E2M1, MXF4 = 0, 1, 2, 3
DTYPES = {"f16": F16, "i8": I8, "e2m1": E2M1, "mxf4": MXF4}
EPILOGUES = {"none": 0, "bias": 1, "gelu": 2, "bias_gelu": 3}
OPS = {"bias": 1, "relu": 2, "gelu": 3, "scale": 4, "clamp": 5, "quant_i8": 6}
MAX_EPILOGUE_OPS = 8
STATUS = {0: "DG_OK", 1: "DG_ERR_INVALID_ARG", 2: "DG_ERR_UNSUPPORTED",
          3: "DG_ERR_NO_VALID_CANDIDATE", 4: "DG_ERR_CUDA", 5: "DG_ERR_TIMEOUT",
          6: "DG_ERR_INVALID_STATE"}
KERNELS = {0: "tc", 1: "gemv", 2: "tc_widened", 3: "skinny", 4: "gemv_mma", 5: "tc_streamk",
           -1: "none"}

# Every symbol include/dg.h declares.
EXPORTS = ["dg_query_hw", "dg_plan_tiles", "dg_gemm", "dg_gemm_planned", "dg_gemm_host",
           "dg_gemm_ex", "dg_gemm_strided_batched", "dg_gemm_grouped",
           "dg_quantize_mxf4", "dg_gemm_mxf4", "dg_gemm_mxf4_planned",
           "dg_gemm_thin_noalloc", "dg_last_error",
           "dg_check_status", "dg_set_wait_timeout_ns", "dg_selftest_wait_timeout",
           "dg_launch_count", "dg_shutdown"]

_HERE = os.path.dirname(os.path.abspath(__file__))


def lib_path():
    return os.path.join(_HERE, "libdg.so")


class DgError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__("%s: %s" % (self.name, message))


class HwDesc(ctypes.Structure):
    _fields_ = [("sm_count", ctypes.c_int), ("cc_major", ctypes.c_int), ("cc_minor", ctypes.c_int),
                ("smem_per_block_optin", ctypes.c_int), ("smem_per_sm", ctypes.c_int),
                ("regs_per_sm", ctypes.c_int), ("regs_per_thread_max", ctypes.c_int),
                ("max_threads_per_sm", ctypes.c_int), ("tmem_cols", ctypes.c_int),
                ("l2_bytes", ctypes.c_int64), ("hbm_gbps", ctypes.c_double),
                ("tc_f16_tflops", ctypes.c_double), ("clock_ghz", ctypes.c_double)]

    def as_dict(self):
        return {f[0]: getattr(self, f[0]) for f in self._fields_}


class TilePlan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("m_tile", ctypes.c_int), ("n_tile", ctypes.c_int),
                ("k_tile", ctypes.c_int), ("split_k", ctypes.c_int), ("stages", ctypes.c_int),
                ("cta_group", ctypes.c_int), ("swap_ab", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("threads", ctypes.c_int),
                ("regs_per_thread", ctypes.c_int), ("grid", ctypes.c_int),
                ("occupancy", ctypes.c_double), ("est_us", ctypes.c_double),
                ("est_tflops", ctypes.c_double)]

    def as_dict(self):
        d = {f[0]: getattr(self, f[0]) for f in self._fields_}
        d["kernel_name"] = KERNELS.get(self.kernel, str(self.kernel))
        return d


_lib = None


class EpilogueOp(ctypes.Structure):
    _fields_ = [("type", ctypes.c_int), ("a", ctypes.c_float), ("b", ctypes.c_float)]


class EpilogueProgram(ctypes.Structure):
    _fields_ = [("n_ops", ctypes.c_int), ("ops", EpilogueOp * MAX_EPILOGUE_OPS)]


def make_program(ops):
    """EpilogueProgram from a list of ops: "relu", "gelu", "bias",
    ("scale", a), ("clamp", lo, hi), ("quant_i8", a) (last op: int8 D), or
    (type_code, a, b)."""
    ops = list(ops)
    if len(ops) > MAX_EPILOGUE_OPS:
        raise ValueError("at most %d epilogue ops" % MAX_EPILOGUE_OPS)
    prog = EpilogueProgram()
    prog.n_ops = len(ops)
    for k, op in enumerate(ops):
        if isinstance(op, str):
            op = (op,)
        code = OPS[op[0]] if isinstance(op[0], str) else int(op[0])
        args = [float(x) for x in op[1:]] + [0.0, 0.0]
        prog.ops[k] = EpilogueOp(code, args[0], args[1])
    return prog


def lib():
    """The loaded libdg.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError("libdg.so is not built (%s); run __graft_entry__.build()" % path)
    L = ctypes.CDLL(path)
    i64, vp, i32, f32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.dg_query_hw.argtypes = [i32, ctypes.POINTER(HwDesc)]
    L.dg_plan_tiles.argtypes = [i64, i64, i64, i32, i32, i32, ctypes.POINTER(HwDesc),
                                ctypes.c_double, ctypes.POINTER(TilePlan), i32,
                                ctypes.POINTER(ctypes.c_int)]
    gemm_args = [i64, i64, i64, i32, i32, vp, i64, vp, i64, vp, vp, f32, f32, i32]
    L.dg_gemm.argtypes = gemm_args + [vp]
    L.dg_gemm_planned.argtypes = gemm_args + [ctypes.POINTER(TilePlan), vp]
    L.dg_gemm_thin_noalloc.argtypes = gemm_args + [vp]
    L.dg_gemm_host.argtypes = [i64, i64, i64, i32, i32, vp, i64, vp, i64, vp, vp, vp, f32, f32,
                               i32, vp]
    L.dg_gemm_strided_batched.argtypes = [i64, i64, i64, i64, i32, i32, vp, i64, i64, vp, i64,
                                          i64, vp, i64, vp, i64, f32, f32, i32, vp]
    L.dg_gemm_grouped.argtypes = [i64, ctypes.POINTER(ctypes.c_int64), i64, i64, i32, i32,
                                  ctypes.POINTER(vp), i64, ctypes.POINTER(vp), i64,
                                  ctypes.POINTER(vp), ctypes.POINTER(vp), f32, f32, i32, vp]
    L.dg_gemm_ex.argtypes = [i64, i64, i64, i32, i32, vp, i64, vp, i64, vp, i64, vp, i64, vp, f32,
                             f32, ctypes.POINTER(EpilogueProgram), vp]
    L.dg_quantize_mxf4.argtypes = [i64, i64, vp, i64, vp, i64, vp, i64, vp]
    L.dg_gemm_mxf4.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp, vp, f32,
                               f32, i32, vp]
    L.dg_gemm_mxf4_planned.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp, vp,
                                       f32, f32, i32, ctypes.POINTER(TilePlan), vp]
    L.dg_last_error.restype = ctypes.c_char_p
    L.dg_last_error.argtypes = []
    L.dg_check_status.argtypes = [vp]
    L.dg_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    L.dg_selftest_wait_timeout.argtypes = [vp]
    L.dg_launch_count.restype = ctypes.c_uint64
    L.dg_launch_count.argtypes = []
    L.dg_shutdown.argtypes = []
    for name in ("dg_query_hw", "dg_plan_tiles", "dg_gemm", "dg_gemm_planned",
                 "dg_gemm_thin_noalloc", "dg_gemm_host", "dg_gemm_ex", "dg_gemm_strided_batched",
                 "dg_gemm_grouped", "dg_quantize_mxf4", "dg_gemm_mxf4", "dg_gemm_mxf4_planned",
                 "dg_check_status",
                 "dg_set_wait_timeout_ns", "dg_selftest_wait_timeout", "dg_shutdown"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def last_error():
    return lib().dg_last_error().decode()


def _check(status):
    if status != 0:
        raise DgError(status, last_error())


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(d):
    return DTYPES[d] if isinstance(d, str) else int(d)


def _epi_code(e):
    return EPILOGUES[e] if isinstance(e, str) else int(e)


def gemm_raw(M, N, K, dtype_a, dtype_b, A, lda, B, ldb, C, bias, alpha, beta, epilogue,
             stream=None, plan=None):
    """dg_gemm / dg_gemm_planned with the C argument order.  A, B, C, bias are
    tensors or raw device addresses; dtypes and epilogue are names or codes."""
    L = lib()
    args = (int(M), int(N), int(K), _dtype_code(dtype_a), _dtype_code(dtype_b), _ptr(A), int(lda),
            _ptr(B), int(ldb), _ptr(C), _ptr(bias), float(alpha), float(beta),
            _epi_code(epilogue))
    s = _stream_handle(stream)
    if plan is None:
        _check(L.dg_gemm(*args, s))
    else:
        _check(L.dg_gemm_planned(*args, ctypes.byref(_as_plan(plan)), s))


_TORCH_DTYPES = None


def _expect(t, kinds, what):
    import torch
    global _TORCH_DTYPES
    if _TORCH_DTYPES is None:
        _TORCH_DTYPES = {"f16": torch.float16, "i8": torch.int8, "e2m1": torch.uint8,
                         "i32": torch.int32}
    if t.dtype != _TORCH_DTYPES[kinds]:
        raise TypeError("%s must be %s, got %s" % (what, _TORCH_DTYPES[kinds], t.dtype))
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("%s must be 2-D with unit column stride" % what)


_TD = None  # (torch, B dtype -> code, code -> torch dtype), built on first use


def _td():
    global _TD
    if _TD is None:
        import torch
        _TD = (torch, {torch.float16: F16, torch.int8: I8, torch.uint8: E2M1},
               (torch.float16, torch.int8, torch.uint8))
    return _TD


def gemm(A, B, C, K=None, bias=None, alpha=1.0, beta=0.0, epilogue="none", dtype_b=None,
         stream=None, plan=None):
    """D = epilogue(alpha * A.B + beta * C), written into C.

    A: [M, lda] (fp16 or int8); B: [N, ldb] (fp16/int8) or [N, ldb/2] uint8
    packed E2M1 codes; C: [M, N] fp16 (int32 for int8); K defaults to
    A.shape[1]; bias: [N] fp16.  The leading dimensions are the row strides.
    (Written for a short host path: small GEMMs are bound by it.)
    """
    torch, b_code, code_dt = _TD or _td()
    da = I8 if A.dtype is torch.int8 else F16
    db = b_code[B.dtype] if dtype_b is None else _dtype_code(dtype_b)
    sa, sb, sc = A.stride(), B.stride(), C.stride()
    names = ("f16", "i8", "e2m1")
    if A.dtype is not code_dt[da] or len(sa) != 2 or sa[1] != 1:
        _expect(A, names[da], "A")
    if B.dtype is not code_dt[db] or len(sb) != 2 or sb[1] != 1:
        _expect(B, names[db], "B")
    if C.dtype is not (torch.int32 if da == I8 else torch.float16) or len(sc) != 2 or sc[1] != 1:
        _expect(C, "i32" if da == I8 else "f16", "C")
    M, N = C.shape
    if A.shape[0] != M or B.shape[0] != N:
        raise ValueError("shape mismatch: A %s, B %s, C %s" % (tuple(A.shape), tuple(B.shape),
                                                               tuple(C.shape)))
    if sc[0] != N:
        raise ValueError("C must be dense row-major (leading dimension N)")
    if K is None:
        K = A.shape[1]
    ldb = sb[0] * (2 if db == E2M1 else 1)
    if plan is not None:
        gemm_raw(M, N, K, da, db, A, sa[0], B, ldb, C, bias, alpha, beta, epilogue,
                 stream=stream, plan=plan)
        return C
    s = _stream_handle(stream)
    _check(lib().dg_gemm(M, N, K, da, db, A.data_ptr(), sa[0], B.data_ptr(), ldb, C.data_ptr(),
                         None if bias is None else bias.data_ptr(), alpha, beta,
                         EPILOGUES[epilogue] if isinstance(epilogue, str) else int(epilogue), s))
    return C


def quantize_mxf4_raw(rows, K, X, ldx, codes, ldq, scales, lds, stream=None):
    """dg_quantize_mxf4 with the C argument order (ldq in codes, lds in bytes)."""
    _check(lib().dg_quantize_mxf4(int(rows), int(K), _ptr(X), int(ldx), _ptr(codes), int(ldq),
                                  _ptr(scales), int(lds), _stream_handle(stream)))


def quantize_mxf4(X, K=None, stream=None):
    """MXFP4 block quantization of the fp16 rows X [rows, >= K] along K.

    Returns (codes, scales): codes uint8 [rows, ldq / 2] (two E2M1 codes per
    byte, ldq = K rounded up to 32), scales uint8 [rows, ceil(K / 32)] (E8M0).
    """
    import torch
    _expect(X, "f16", "X")
    rows = X.shape[0]
    K = X.shape[1] if K is None else int(K)
    ldq = (K + 31) // 32 * 32
    nblk = (K + 31) // 32
    codes = torch.zeros((rows, ldq // 2), dtype=torch.uint8, device=X.device)
    scales = torch.zeros((rows, nblk), dtype=torch.uint8, device=X.device)
    quantize_mxf4_raw(rows, K, X, X.stride(0), codes, ldq, scales, nblk, stream)
    return codes, scales


def _as_plan(plan):
    if isinstance(plan, dict):
        return TilePlan(**{k: v for k, v in plan.items() if k in dict(TilePlan._fields_)})
    return plan


def gemm_mxf4_raw(M, N, K, A, lda, scale_a, lds_a, B, ldb, scale_b, lds_b, C, bias, alpha, beta,
                  epilogue="none", stream=None, plan=None):
    """dg_gemm_mxf4 (dg_gemm_mxf4_planned with a plan) with the C argument
    order (lda, ldb in codes)."""
    epi = EPILOGUES[epilogue] if isinstance(epilogue, str) else int(epilogue)
    args = (int(M), int(N), int(K), _ptr(A), int(lda), _ptr(scale_a), int(lds_a), _ptr(B),
            int(ldb), _ptr(scale_b), int(lds_b), _ptr(C), _ptr(bias), float(alpha), float(beta),
            epi)
    if plan is None:
        _check(lib().dg_gemm_mxf4(*args, _stream_handle(stream)))
    else:
        _check(lib().dg_gemm_mxf4_planned(*args, ctypes.byref(_as_plan(plan)),
                                          _stream_handle(stream)))


def gemm_mxf4(A, scale_a, B, scale_b, C, K, bias=None, alpha=1.0, beta=0.0, epilogue="none",
              stream=None, plan=None):
    """D = epilogue(alpha * A.B + beta * C) for MXFP4 A and B, written into C.

    A: uint8 [M, lda / 2] packed codes with scale_a uint8 [M, >= ceil(K/32)];
    B: uint8 [N, ldb / 2] with scale_b [N, ...]; C: fp16 [M, N] dense.
    plan: a dg_plan_tiles candidate for (M, N, K, "mxf4", "mxf4") to run
    instead of the planner's first.
    """
    for t, what in ((A, "A"), (B, "B"), (scale_a, "scale_a"), (scale_b, "scale_b")):
        _expect(t, "e2m1", what)
    _expect(C, "f16", "C")
    M, N = C.shape
    if A.shape[0] != M or B.shape[0] != N or scale_a.shape[0] != M or scale_b.shape[0] != N:
        raise ValueError("shape mismatch")
    if C.stride(0) != N:
        raise ValueError("C must be dense row-major (leading dimension N)")
    gemm_mxf4_raw(M, N, K, A, 2 * A.stride(0), scale_a, scale_a.stride(0), B, 2 * B.stride(0),
                  scale_b, scale_b.stride(0), C, bias, alpha, beta, epilogue, stream, plan)
    return C


def gemm_ex_raw(M, N, K, dtype_a, dtype_b, A, lda, B, ldb, C, ldc, D, ldd, bias, alpha, beta,
                program=None, stream=None):
    """dg_gemm_ex with the C argument order.  program: None, an
    EpilogueProgram, or a list of ops for make_program."""
    if program is not None and not isinstance(program, EpilogueProgram):
        program = make_program(program)
    args = (int(M), int(N), int(K), _dtype_code(dtype_a), _dtype_code(dtype_b), _ptr(A), int(lda),
            _ptr(B), int(ldb), _ptr(C), int(ldc), _ptr(D), int(ldd), _ptr(bias), float(alpha),
            float(beta), ctypes.byref(program) if program is not None else None,
            _stream_handle(stream))
    _check(lib().dg_gemm_ex(*args))


def gemm_ex(A, B, D, C=None, K=None, bias=None, alpha=1.0, beta=0.0, program=(), dtype_b=None,
            stream=None):
    """D = program(alpha * A.B + beta * C) with C read and D written.

    A and B as in gemm(); C and D are [M, N] views with unit column stride
    and any row stride (leading dimension) >= N, e.g. column slices of wider
    buffers; C may be D itself.  program: list of ops, applied in order
    ("bias", "relu", "gelu", ("scale", a), ("clamp", lo, hi)); a program
    ending in ("quant_i8", a) writes an int8 D (C, when given, stays fp16).
    """
    import torch
    dtype_a = "i8" if A.dtype == torch.int8 else "f16"
    if dtype_b is None:
        dtype_b = {torch.float16: "f16", torch.int8: "i8", torch.uint8: "e2m1"}[B.dtype]
    _expect(A, dtype_a, "A")
    _expect(B, dtype_b, "B")
    out = "i32" if dtype_a == "i8" else "f16"
    ops = list(program or [])
    last = ops[-1] if ops else None
    quant = last is not None and (last[0] if isinstance(last, tuple) else last) in ("quant_i8", 6)
    _expect(D, "i8" if quant else out, "D")
    M, N = D.shape
    ldc = D.stride(0)
    if C is not None:
        _expect(C, out, "C")
        if tuple(C.shape) != (M, N):
            raise ValueError("C must be [M, N] like D")
        ldc = C.stride(0)
    if A.shape[0] != M or B.shape[0] != N:
        raise ValueError("shape mismatch: A %s, B %s, D %s" % (tuple(A.shape), tuple(B.shape),
                                                               tuple(D.shape)))
    if K is None:
        K = A.shape[1]
    ldb = B.stride(0) * (2 if dtype_b == "e2m1" else 1)
    gemm_ex_raw(M, N, K, dtype_a, dtype_b, A, A.stride(0), B, ldb, C, ldc, D, D.stride(0), bias,
                alpha, beta, program=make_program(ops), stream=stream)
    return D


def gemm_strided_batched_raw(batch, M, N, K, dtype_a, dtype_b, A, lda, stride_a, B, ldb, stride_b,
                             C, stride_c, bias, stride_bias, alpha, beta, epilogue, stream=None):
    """dg_gemm_strided_batched with the C argument order."""
    args = (int(batch), int(M), int(N), int(K), _dtype_code(dtype_a), _dtype_code(dtype_b),
            _ptr(A), int(lda), int(stride_a), _ptr(B), int(ldb), int(stride_b), _ptr(C),
            int(stride_c), _ptr(bias), int(stride_bias), float(alpha), float(beta),
            _epi_code(epilogue), _stream_handle(stream))
    _check(lib().dg_gemm_strided_batched(*args))


def gemm_batched(A, B, C, K=None, bias=None, alpha=1.0, beta=0.0, epilogue="none",
                 dtype_b=None, stream=None):
    """D_z = epilogue(alpha * A_z.B_z + beta * C_z) for every z, written into C.

    A: [batch, M, lda]; B: [batch, N, ldb] or [N, ldb] (shared by all
    problems; uint8 packed codes for E2M1); C: [batch, M, N], each [M, N]
    dense; bias: [batch, N] or [N] (shared).  The batch strides are the
    tensors' first-dimension strides.
    """
    import torch
    dtype_a = "i8" if A.dtype == torch.int8 else "f16"
    if dtype_b is None:
        dtype_b = {torch.float16: "f16", torch.int8: "i8", torch.uint8: "e2m1"}[B.dtype]
    if A.dim() != 3 or C.dim() != 3 or B.dim() not in (2, 3):
        raise ValueError("A and C must be 3-D, B 2-D or 3-D")
    batch, M, N = C.shape
    _expect(A[0], dtype_a, "A")
    B0 = B[0] if B.dim() == 3 else B
    _expect(B0, dtype_b, "B")
    _expect(C[0], "i32" if dtype_a == "i8" else "f16", "C")
    if A.shape[0] != batch or A.shape[1] != M or B0.shape[0] != N or \
            (B.dim() == 3 and B.shape[0] != batch):
        raise ValueError("shape mismatch: A %s, B %s, C %s" % (tuple(A.shape), tuple(B.shape),
                                                               tuple(C.shape)))
    if C.stride(1) != N:
        raise ValueError("each C[z] must be dense row-major (leading dimension N)")
    if K is None:
        K = A.shape[2]
    codes = 2 if dtype_b == "e2m1" else 1
    ldb = B0.stride(0) * codes
    stride_b = B.stride(0) * codes if B.dim() == 3 else 0
    stride_bias = 0
    if bias is not None and bias.dim() == 2:
        stride_bias = bias.stride(0)
    gemm_strided_batched_raw(batch, M, N, K, dtype_a, dtype_b, A, A.stride(1), A.stride(0), B,
                             ldb, stride_b, C, C.stride(0), bias, stride_bias, alpha, beta,
                             epilogue, stream=stream)
    return C


def prepare_grouped(As, Bs, Cs, K=None, bias=None, alpha=1.0, beta=0.0, epilogue="none"):
    """Checks a group of problems once and returns run(stream=None), which
    issues dg_gemm_grouped on them with the prepared pointer arrays (for a
    group that is run again and again, e.g. one mixture-of-experts layer).
    The tensors must stay alive and keep their storage.  Arguments as
    gemm_grouped."""
    import torch
    count = len(As)
    if not isinstance(Bs, (list, tuple)):
        Bs = [Bs] * count
    if bias is not None and not isinstance(bias, (list, tuple)):
        bias = [bias] * count
    if len(Bs) != count or len(Cs) != count or (bias is not None and len(bias) != count):
        raise ValueError("As, Bs, Cs (and bias) must have one entry per problem")
    if count == 0:
        return lambda stream=None: Cs
    A0, B0 = As[0], Bs[0]
    dtype_a = "i8" if A0.dtype == torch.int8 else "f16"
    dtype_b = {torch.float16: "f16", torch.int8: "i8", torch.uint8: "e2m1"}[B0.dtype]
    N = Cs[0].shape[1]
    if K is None:
        K = A0.shape[1]
    lda = A0.stride(0)
    ldb = B0.stride(0) * (2 if dtype_b == "e2m1" else 1)
    for g in range(count):
        _expect(As[g], dtype_a, "A[%d]" % g)
        _expect(Bs[g], dtype_b, "B[%d]" % g)
        _expect(Cs[g], "i32" if dtype_a == "i8" else "f16", "C[%d]" % g)
        if As[g].stride(0) != lda or Bs[g].stride(0) * (2 if dtype_b == "e2m1" else 1) != ldb:
            raise ValueError("every problem must share lda and ldb")
        if Cs[g].shape[1] != N or Cs[g].shape[0] != As[g].shape[0] or Bs[g].shape[0] != N or \
                (Cs[g].shape[0] and Cs[g].stride(0) != N):
            raise ValueError("problem %d: shapes or C layout do not match" % g)
    vp = ctypes.c_void_p
    Ms = (ctypes.c_int64 * count)(*[int(a.shape[0]) for a in As])
    pa = (vp * count)(*[a.data_ptr() for a in As])
    pb = (vp * count)(*[b.data_ptr() for b in Bs])
    pc = (vp * count)(*[c.data_ptr() for c in Cs])
    pbias = None if bias is None else (vp * count)(*[b.data_ptr() for b in bias])
    args = (count, Ms, int(N), int(K), _dtype_code(dtype_a), _dtype_code(dtype_b), pa, int(lda),
            pb, int(ldb), pc, pbias, float(alpha), float(beta), _epi_code(epilogue))
    fn = lib().dg_gemm_grouped

    def run(stream=None):
        _check(fn(*args, _stream_handle(stream)))
        return Cs
    return run


def gemm_grouped(As, Bs, Cs, K=None, bias=None, alpha=1.0, beta=0.0, epilogue="none",
                 stream=None):
    """D_g = epilogue(alpha * A_g.B_g + beta * C_g) for every g, written into Cs[g].

    As: list of [M_g, lda] tensors (one lda, M_g may differ, 0 skips); Bs: a
    list of [N, ldb] tensors or one tensor shared by all; Cs: list of [M_g, N]
    dense tensors; bias: None, one [N] tensor or a list.  All problems share
    N, K, the dtypes, scalars and epilogue.
    """
    return prepare_grouped(As, Bs, Cs, K, bias, alpha, beta, epilogue)(stream)
    A0, B0 = As[0], Bs[0]
    dtype_a = "i8" if A0.dtype == torch.int8 else "f16"
    dtype_b = {torch.float16: "f16", torch.int8: "i8", torch.uint8: "e2m1"}[B0.dtype]
    N = Cs[0].shape[1]
    if K is None:
        K = A0.shape[1]
    lda = A0.stride(0)
    ldb = B0.stride(0) * (2 if dtype_b == "e2m1" else 1)
    for g in range(count):
        _expect(As[g], dtype_a, "A[%d]" % g)
        _expect(Bs[g], dtype_b, "B[%d]" % g)
        _expect(Cs[g], "i32" if dtype_a == "i8" else "f16", "C[%d]" % g)
        if As[g].stride(0) != lda or Bs[g].stride(0) * (2 if dtype_b == "e2m1" else 1) != ldb:
            raise ValueError("every problem must share lda and ldb")
        if Cs[g].shape[1] != N or Cs[g].shape[0] != As[g].shape[0] or Bs[g].shape[0] != N or \
                (Cs[g].shape[0] and Cs[g].stride(0) != N):
            raise ValueError("problem %d: shapes or C layout do not match" % g)
    vp = ctypes.c_void_p
    Ms = (ctypes.c_int64 * count)(*[int(a.shape[0]) for a in As])
    pa = (vp * count)(*[a.data_ptr() for a in As])
    pb = (vp * count)(*[b.data_ptr() for b in Bs])
    pc = (vp * count)(*[c.data_ptr() for c in Cs])
    pbias = None if bias is None else (vp * count)(*[b.data_ptr() for b in bias])
    _check(lib().dg_gemm_grouped(count, Ms, int(N), int(K), _dtype_code(dtype_a),
                                 _dtype_code(dtype_b), pa, int(lda), pb, int(ldb), pc, pbias,
                                 float(alpha), float(beta), _epi_code(epilogue),
                                 _stream_handle(stream)))
    return Cs


def gemm_host_raw(M, N, K, dtype_a, dtype_b, A, lda, B, ldb, C, D, bias, alpha, beta, epilogue,
                  stream=None):
    """dg_gemm_host with the C argument order: A, B, C, D, bias are host
    tensors (ideally pinned) or raw host addresses."""
    args = (int(M), int(N), int(K), _dtype_code(dtype_a), _dtype_code(dtype_b), _ptr(A), int(lda),
            _ptr(B), int(ldb), _ptr(C), _ptr(D), _ptr(bias), float(alpha), float(beta),
            _epi_code(epilogue), _stream_handle(stream))
    _check(lib().dg_gemm_host(*args))


def gemm_host(A, B, D, C=None, K=None, bias=None, alpha=1.0, beta=0.0, epilogue="none",
              dtype_b=None, stream=None):
    """D = epilogue(alpha * A.B + beta * C) on host (CPU) tensors, copies
    included: the call is asynchronous on `stream`, so synchronise it before
    reading D.  Layouts as gemm(); C (read when beta != 0) and D are [M, N]."""
    import torch
    dtype_a = "i8" if A.dtype == torch.int8 else "f16"
    if dtype_b is None:
        dtype_b = {torch.float16: "f16", torch.int8: "i8", torch.uint8: "e2m1"}[B.dtype]
    for t, what in ((A, "A"), (B, "B"), (D, "D"), (C, "C"), (bias, "bias")):
        if t is not None and t.device.type != "cpu":
            raise ValueError("%s must be a host tensor" % what)
    _expect(A, dtype_a, "A")
    _expect(B, dtype_b, "B")
    out = "i32" if dtype_a == "i8" else "f16"
    _expect(D, out, "D")
    M, N = D.shape
    if C is not None:
        _expect(C, out, "C")
        if tuple(C.shape) != (M, N) or C.stride(0) != N:
            raise ValueError("C must be dense [M, N]")
    if A.shape[0] != M or B.shape[0] != N or D.stride(0) != N:
        raise ValueError("shape mismatch: A %s, B %s, D %s" % (tuple(A.shape), tuple(B.shape),
                                                               tuple(D.shape)))
    if K is None:
        K = A.shape[1]
    ldb = B.stride(0) * (2 if dtype_b == "e2m1" else 1)
    gemm_host_raw(M, N, K, dtype_a, dtype_b, A, A.stride(0), B, ldb, C, D, bias, alpha, beta,
                  epilogue, stream=stream)
    return D


def query_hw(device=0):
    h = HwDesc()
    _check(lib().dg_query_hw(int(device), ctypes.byref(h)))
    return h


def plan_tiles(M, N, K, dtype_a="f16", dtype_b="f16", epilogue="none", hw=None,
               target_occupancy=0.0, max_out=64):
    """The planner's ranked candidates (list of dicts)."""
    if isinstance(hw, dict):
        h = HwDesc(**hw)
        hw_p = ctypes.byref(h)
    elif hw is not None:
        hw_p = ctypes.byref(hw)
    else:
        hw_p = None
    out = (TilePlan * max_out)()
    n = ctypes.c_int(0)
    _check(lib().dg_plan_tiles(int(M), int(N), int(K), _dtype_code(dtype_a), _dtype_code(dtype_b),
                               _epi_code(epilogue), hw_p, float(target_occupancy), out,
                               int(max_out), ctypes.byref(n)))
    return [out[i].as_dict() for i in range(n.value)]


def check_status(stream=None):
    _check(lib().dg_check_status(_stream_handle(stream)))


def set_wait_timeout_ns(ns):
    _check(lib().dg_set_wait_timeout_ns(int(ns)))


def selftest_wait_timeout(stream=None):
    _check(lib().dg_selftest_wait_timeout(_stream_handle(stream)))


def launch_count():
    return int(lib().dg_launch_count())


def shutdown():
    _check(lib().dg_shutdown())
