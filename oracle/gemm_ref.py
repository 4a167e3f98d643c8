"""Plain fp64 / exact-integer definition of D = epilogue(alpha * A.B^T + beta * C).

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path.

Operand conventions (the same ones the C ABI uses, stated here on their own):
  * A is the M x K activation matrix.
  * B is given as N rows of K (each output column j owns one contiguous row of
    B), so the product is  acc[i, j] = sum_k A[i, k] * B[j, k].
  * C and D are M x N.

Functions and what each follows:
  e2m1_value / e2m1_decode -- 4-bit weight code of the discosf.com "DeepGEMM"
      article, section 2.2 layer 2: 2 exponent bits + 1 mantissa bit (+ sign),
      magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}.  Pinned by a code table typed
      from the format definition (tests/golden/e2m1_codes.txt).
  unpack_e2m1 -- two codes per byte (same article, section 4.3, "pack_int4");
      the pages do not fix the nibble order.  Reading taken: byte p of a
      column's row holds k = 2p in its low nibble and k = 2p+1 in its high
      nibble.  Pinned by a hand-built byte vector.
  gelu_erf -- the GELU of the fused epilogue (kwkr.cn "DeepGEMM" article,
      section 2.2 third layer; discosf.com article section 6.1), exact erf
      form x * Phi(x).  Pinned by printed normal-CDF table values and identities.
  gemm_reference -- the definition itself: exact products, fp64 (or exact
      integer) sums, then t = alpha*acc + beta*C + bias, then GELU if asked.
      Epilogue order (bias after alpha/beta, before GELU) is the reading of
      kwkr.cn section 2.2 third layer + section 3.2 step 3.  Pinned by closed
      forms (identity, permutation, all-ones, rank-1, int8 extremes) and by
      exact rational brute force on tiny shapes.
  apply_program -- an epilogue program: ops applied in order to t (the
      op_type registry of the fused epilogue, kwkr.cn section 2.2 third layer:
      bias add, ReLU, quantization-style scale and saturation; discosf.com
      section 6.1: GELU chosen by op type).  Reading taken: each op is the
      plain real function (t + bias_j, max(t, 0), GELU, a * t, min(max(t, lo),
      hi)); the op operands a, lo, hi are binary32 numbers, the type the C ABI
      passes them in.  "quant_i8" (last op only) is the output quantization of
      the same passage: D becomes int8, round-half-to-even(a * t) saturated to
      [-128, 127], NaN to 0.  Pinned by hand-computed values and
      order-sensitivity cases.
  error_bound -- the floating-point acceptance bound
      2^-10 * (|A|.|B|)_ij + 2^-10 * |D_ref|_ij, with (|A|.|B|) read as the
      magnitude of every term that enters t, a 2^-24 floor, and a GELU
      Lipschitz factor; for a program, the input error carried through each
      op by its Lipschitz constant, and |a| E + 1 for an int8 quantization
      (the error of a * t, plus half a unit for each side's rounding).  Pinned
      by direct checks on hand-computed cases.
"""

import math

import numpy as np

# Field widths of one E2M1 code: sign, exponent, mantissa (bit 3 | bits 2..1 | bit 0).
E2M1_BITS = (1, 2, 1)

# max |d/dx GELU(x)| over the real line is 1.1289 (at x = sqrt(2)); 1.13 bounds it.
GELU_LIPSCHITZ = 1.13

_EPILOGUES = ("none", "bias", "gelu", "bias_gelu")

# Ops of an epilogue program and the number of operands each takes.
PROGRAM_OPS = {"bias": 0, "relu": 0, "gelu": 0, "scale": 1, "clamp": 2, "quant_i8": 1}


def e2m1_value(code):
    """Real value of one 4-bit E2M1 code.

    Exponent field e (bias 1) and mantissa bit m: e == 0 is the subnormal
    range, value 0.5*m; otherwise 2^(e-1) * (1 + m/2).  The sign bit negates
    (code 8 is -0.0).
    """
    code = int(code)
    if not 0 <= code <= 15:
        raise ValueError("E2M1 code out of range: %r" % code)
    sign = (code >> 3) & 1
    exp = (code >> 1) & 3
    man = code & 1
    if exp == 0:
        mag = 0.5 * man
    else:
        mag = math.ldexp(1.0 + 0.5 * man, exp - 1)
    return -mag if sign else mag


_E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def e2m1_decode(codes):
    """Decode an integer array of 4-bit codes to float64 values."""
    codes = np.asarray(codes)
    if codes.size and (codes.min() < 0 or codes.max() > 15):
        raise ValueError("E2M1 codes must lie in [0, 15]")
    return _E2M1_TABLE[codes.astype(np.int64)]


def unpack_e2m1(packed, K):
    """Split packed bytes [N, nbytes] into codes [N, K].

    Byte p of a row carries k = 2p (low nibble) and k = 2p + 1 (high nibble).
    """
    packed = np.asarray(packed, dtype=np.uint8)
    if packed.ndim != 2:
        raise ValueError("packed weights must be 2-D [N, bytes]")
    if 2 * packed.shape[1] < K:
        raise ValueError("packed rows hold %d codes, need K=%d" % (2 * packed.shape[1], K))
    codes = np.empty((packed.shape[0], 2 * packed.shape[1]), dtype=np.uint8)
    codes[:, 0::2] = packed & 0x0F
    codes[:, 1::2] = packed >> 4
    return codes[:, :K]


def _erf(x):
    try:
        from scipy.special import erf  # vectorised, double precision
        return erf(x)
    except ImportError:  # pragma: no cover - scipy is present on both hosts
        return np.vectorize(math.erf, otypes=[np.float64])(x)


def gelu_erf(t):
    """GELU(t) = 0.5 * t * (1 + erf(t / sqrt(2))) in float64."""
    t = np.asarray(t, dtype=np.float64)
    return 0.5 * t * (1.0 + _erf(t / math.sqrt(2.0)))


def _normalise_program(program):
    """[(name, operands...)] with binary32-rounded operands, validated."""
    out = []
    for op in program:
        if isinstance(op, str):
            op = (op,)
        name, args = op[0], tuple(op[1:])
        if name not in PROGRAM_OPS:
            raise ValueError("unknown epilogue op %r" % (name,))
        if len(args) != PROGRAM_OPS[name]:
            raise ValueError("op %r takes %d operands" % (name, PROGRAM_OPS[name]))
        args = tuple(float(np.float32(x)) for x in args)
        if name == "clamp" and not args[0] <= args[1]:
            raise ValueError("clamp needs lo <= hi")
        out.append((name,) + args)
    if any(op[0] == "quant_i8" for op in out[:-1]):
        raise ValueError("quant_i8 must be the last op")
    return out


def quantize_i8(x):
    """Round half to even, saturate to [-128, 127]; NaN to 0 (float64 codes)."""
    x = np.asarray(x, dtype=np.float64)
    q = np.clip(np.rint(np.nan_to_num(x, nan=0.0, posinf=np.inf, neginf=-np.inf)), -128, 127)
    return np.where(np.isnan(x), 0.0, q)


def apply_program(t, program, bias=None):
    """The epilogue program's ops, in order, on t (float64, [rows, N]).

    bias (float16 [N]) is read by the "bias" op: t_ij + bias_j.
    """
    t = np.asarray(t, dtype=np.float64)
    for op in _normalise_program(program):
        name = op[0]
        if name == "bias":
            if bias is None:
                raise ValueError("a bias op needs a bias vector")
            bias = np.asarray(bias)
            if bias.dtype != np.float16:
                raise TypeError("bias must be float16")
            t = t + bias.astype(np.float64)[None, :]
        elif name == "relu":
            t = np.where(t > 0.0, t, 0.0)
        elif name == "gelu":
            t = gelu_erf(t)
        elif name == "scale":
            t = op[1] * t
        elif name == "clamp":
            t = np.minimum(np.maximum(t, op[1]), op[2])
        else:  # quant_i8
            t = quantize_i8(op[1] * t)
    return t


def _operand_a(A, dtype_a):
    if dtype_a == "f16":
        A = np.asarray(A)
        if A.dtype != np.float16:
            raise TypeError("f16 operand A must be float16")
        return A.astype(np.float64)
    if dtype_a == "i8":
        A = np.asarray(A)
        if A.dtype != np.int8:
            raise TypeError("i8 operand A must be int8")
        return A.astype(np.float64)
    raise ValueError("unsupported dtype for A: %r" % (dtype_a,))


def _operand_b(B, dtype_b, K):
    if dtype_b == "f16":
        B = np.asarray(B)
        if B.dtype != np.float16:
            raise TypeError("f16 operand B must be float16")
        return B[:, :K].astype(np.float64)
    if dtype_b == "i8":
        B = np.asarray(B)
        if B.dtype != np.int8:
            raise TypeError("i8 operand B must be int8")
        return B[:, :K].astype(np.float64)
    if dtype_b == "e2m1":
        return e2m1_decode(unpack_e2m1(B, K))
    raise ValueError("unsupported dtype for B: %r" % (dtype_b,))


def _check_pair(dtype_a, dtype_b):
    if (dtype_a, dtype_b) not in (("f16", "f16"), ("i8", "i8"), ("f16", "e2m1")):
        raise ValueError("unsupported dtype pair %r x %r" % (dtype_a, dtype_b))


def _wrap_int32(x_u64):
    """Low 32 bits of a uint64 array, read as two's-complement int32."""
    return (x_u64 & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.int32).astype(np.int64)


def gemm_reference(A, B, K, dtype_a="f16", dtype_b="f16", C=None, bias=None,
                   alpha=1.0, beta=0.0, epilogue="none", rows=None, program=None):
    """D_ref for every row (or only for ``rows``) of the output.

    Floating-point pairs return float64 (no output rounding).  The int8 pair
    returns int64 values in the int32 range: the exact integer sum, then
    alpha*acc + beta*C taken modulo 2^32 (alpha and beta must be integers).
    ``program`` (a list of ops, see apply_program) replaces ``epilogue``:
    D = program(alpha*acc + beta*C).
    """
    _check_pair(dtype_a, dtype_b)
    if epilogue not in _EPILOGUES:
        raise ValueError("unknown epilogue %r" % (epilogue,))
    if program and epilogue != "none":
        raise ValueError("give an epilogue or a program, not both")
    A = np.asarray(A)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        A = A[rows]
        if C is not None:
            C = np.asarray(C)[rows]
    a = _operand_a(A[:, :K], dtype_a)
    b = _operand_b(B, dtype_b, K)
    # Every product of two fp16 values (or of an fp16 value and an E2M1 value,
    # or of two int8 values) is exact in float64; the fp64 sum of K of them
    # carries a relative error of at most about K * 2^-53.
    acc = a @ b.T

    if dtype_a == "i8":
        if epilogue != "none" or bias is not None or program:
            raise ValueError("the int8 path has no bias/GELU epilogue or program")
        if float(alpha) != int(alpha) or float(beta) != int(beta):
            raise ValueError("the int8 path takes integral alpha and beta")
        # |acc| <= K * 2^14, an integer below 2^53 for K < 2^39, hence exact.
        acc_i = acc.astype(np.int64)
        mod = 1 << 64
        t = np.uint64(int(alpha) % mod) * acc_i.astype(np.uint64)
        if beta != 0:
            if C is None:
                raise ValueError("beta != 0 needs C")
            c_u = np.asarray(C, dtype=np.int32).astype(np.int64).astype(np.uint64)
            t = t + np.uint64(int(beta) % mod) * c_u
        return _wrap_int32(t)

    return fp_epilogue(acc, C, bias, alpha, beta, epilogue, program)


def fp_epilogue(acc, C, bias, alpha, beta, epilogue, program):
    """The floating-point epilogue on the exact products' sums acc (float64):
    t = alpha*acc + beta*C, then the program, or bias and GELU."""
    if epilogue not in _EPILOGUES:
        raise ValueError("unknown epilogue %r" % (epilogue,))
    if program and epilogue != "none":
        raise ValueError("give an epilogue or a program, not both")
    t = float(alpha) * acc
    if beta != 0.0:
        if C is None:
            raise ValueError("beta != 0 needs C")
        C = np.asarray(C)
        if C.dtype != np.float16:
            raise TypeError("C must be float16 on the floating-point paths")
        t = t + float(beta) * C.astype(np.float64)
    if program:
        return apply_program(t, program, bias)
    if epilogue in ("bias", "bias_gelu"):
        if bias is None:
            raise ValueError("bias epilogue needs a bias vector")
        bias = np.asarray(bias)
        if bias.dtype != np.float16:
            raise TypeError("bias must be float16")
        t = t + bias.astype(np.float64)[None, :]
    if epilogue in ("gelu", "bias_gelu"):
        return gelu_erf(t)
    return t


def error_bound(A, B, K, D_ref, dtype_a="f16", dtype_b="f16", C=None, bias=None,
                alpha=1.0, beta=0.0, epilogue="none", rows=None, program=None):
    """Per-element acceptance bound for floating-point results.

    bound = g * 2^-10 * P_ij + 2^-10 * |D_ref|_ij + 2^-24, where
      P_ij = |alpha| * sum_k |A_ik| |B_jk| + |beta| |C_ij| + |bias_j|
    is the magnitude of everything that enters the pre-activation t, g = 1
    without GELU and g = GELU_LIPSCHITZ with it (an error in t moves GELU(t)
    by at most that factor), and 2^-24 (the smallest fp16 subnormal) lets
    exact zeros and fp16-subnormal outputs compare.

    With a program, E = 2^-10 * P_0 (P_0 without the bias) is the error
    allowed in t on entry and each op carries it forward: a bias op adds
    2^-10 |bias_j|, GELU multiplies it by GELU_LIPSCHITZ, scale by |a|, ReLU
    and clamp (Lipschitz 1) keep it; every op adds 2^-20 |t| after it for the
    binary32 rounding of that op.  bound = E + 2^-10 |D_ref| + 2^-24.
    """
    _check_pair(dtype_a, dtype_b)
    A = np.asarray(A)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        A = A[rows]
        if C is not None:
            C = np.asarray(C)[rows]
    return fp_bound(_operand_a(A[:, :K], dtype_a), _operand_b(B, dtype_b, K), D_ref, C, bias,
                    alpha, beta, epilogue, program)


def fp_bound(a, b, D_ref, C, bias, alpha, beta, epilogue, program):
    """error_bound's formula on decoded operands a [rows, K] and b [N, K]."""
    P = abs(float(alpha)) * (np.abs(a) @ np.abs(b).T)
    if beta != 0.0 and C is not None:
        P = P + abs(float(beta)) * np.abs(np.asarray(C).astype(np.float64))
    if program:
        # t on entry, recomputed from its definition to track |t| per op
        t = float(alpha) * (a @ b.T)
        if beta != 0.0 and C is not None:
            t = t + float(beta) * np.asarray(C).astype(np.float64)
        E = 2.0 ** -10 * P
        for op in _normalise_program(program):
            name = op[0]
            if name == "bias":
                E = E + 2.0 ** -10 * np.abs(np.asarray(bias).astype(np.float64))[None, :]
            elif name == "gelu":
                E = GELU_LIPSCHITZ * E
            elif name == "scale":
                E = abs(op[1]) * E
            elif name == "quant_i8":
                E = abs(op[1]) * E + 1.0
            t = apply_program(t, [op], bias)
            if name != "quant_i8":
                E = E + 2.0 ** -20 * np.abs(t)
        return E + 2.0 ** -10 * np.abs(D_ref) + 2.0 ** -24
    if epilogue in ("bias", "bias_gelu") and bias is not None:
        P = P + np.abs(np.asarray(bias).astype(np.float64))[None, :]
    g = GELU_LIPSCHITZ if epilogue in ("gelu", "bias_gelu") else 1.0
    return g * 2.0 ** -10 * P + 2.0 ** -10 * np.abs(D_ref) + 2.0 ** -24
