"""Plain definition of block-scaled 4-bit operands (MXFP4) and of the GEMM on them.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path.

What the pages fix and what is read into them
  The discosf.com "DeepGEMM" article (section 2.2 layer 2, section 4.3) asks
  for low-bit operands in the tensor cores' own formats, with the weight code
  int4_e2m1 (2 exponent bits, 1 mantissa bit), rather than an FP16 emulation.
  It names no block size and no scale format.  Reading taken: the MX block
  format that block-scaled tensor-core MMAs consume (OCP Microscaling Formats
  v1.0, the MXFP4 type), stated here in our own words:

  * A block is 32 consecutive values of one row along K (the last block of a
    row holds K mod 32 values when K is not a multiple of 32).
  * Each block carries one scale X = 2^s, stored as an E8M0 byte: the 8-bit
    unsigned exponent e = s + 127, e in [0, 254]; e = 255 means NaN.
  * Each value carries one E2M1 code P (sign, 2 exponent bits, 1 mantissa
    bit; magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}; gemm_ref.e2m1_value).
    The value the pair stands for is e2m1(P) * X.

  Quantization of a block of real values V_1..V_n (mxfp4_quantize):
    1. amax = max |V_i|.
    2. s = floor(log2(amax)) - 2, where 2 is the exponent of E2M1's largest
       power of two (4 = 2^2; the largest code is 6 = 1.5 * 2^2), clamped to
       [-127, 127]; an all-zero block takes s = -127 (the clamp of -inf).
    3. P_i = V_i / 2^s rounded to the nearest E2M1 magnitude, ties to the
       code with mantissa bit 0, saturated at 6 (values in (6, 8) become 6),
       with the sign of V_i kept (a negative value that rounds to zero gives
       the -0 code, 8).
    4. A block holding a NaN or an infinity gets e = 255 and codes 0.

  The GEMM (gemm_mx_reference): A is M x K and B is N rows of K, both as
  MXFP4 (packed codes, two per byte, low nibble = even k, the packing of the
  E2M1 weights; plus an E8M0 byte per block).  acc_ij = sum_k a_ik b_jk with
  a = e2m1(P) * X exactly (float64 holds every such value and product), then
  the same epilogue as the FP16 path: t = alpha acc + beta C + bias, GELU or a
  program.  The kernel accumulates in FP32, so the floating-point acceptance
  bound is the FP16 path's one with |a|, |b| the decoded operands.

Parity pins (tests/test_oracle_mx.py): E8M0 values typed from the format
definition (tests/golden/e8m0_values.txt), brute-force nearest-code search
over the 15 representable values for the rounding, closed forms for the
scale (exact powers of two, values just below one), exact reconstruction of
blocks that are already on the grid, the non-finite and all-zero blocks,
ragged last blocks, and exact rational brute force for the GEMM; planted
mistakes (wrong exponent offset, ceil for floor, ties away from zero, no
saturation, lost signs, 16-value blocks, row-wide scales) each fail a pin.
"""

import math

import numpy as np

from . import gemm_ref

MX_BLOCK = 32          # values per scale block
E2M1_EMAX = 2          # exponent of the largest power of two E2M1 holds
E8M0_BIAS = 127
E8M0_NAN = 255

# E2M1 magnitudes by 3-bit magnitude code (sign bit excluded)
_MAGS = np.array([gemm_ref.e2m1_value(c) for c in range(8)], dtype=np.float64)


def e8m0_value(code):
    """Real value of one E8M0 scale byte: 2^(code - 127); 255 is NaN."""
    code = int(code)
    if not 0 <= code <= 255:
        raise ValueError("E8M0 code out of range: %r" % code)
    if code == E8M0_NAN:
        return float("nan")
    return math.ldexp(1.0, code - E8M0_BIAS)


def e8m0_decode(codes):
    codes = np.asarray(codes, dtype=np.int64)
    out = np.ldexp(1.0, codes - E8M0_BIAS)
    return np.where(codes == E8M0_NAN, np.nan, out)


def e2m1_round(q):
    """E2M1 codes (0..15) of the real values q (float64): nearest magnitude,
    ties to the even mantissa bit, saturated at 6, sign kept."""
    q = np.asarray(q, dtype=np.float64)
    m = np.abs(q)
    # each midpoint between neighbours; at a tie the neighbour whose code is
    # even (mantissa bit 0) wins
    code = np.zeros(m.shape, dtype=np.int64)
    for c in range(7):
        mid = 0.5 * (_MAGS[c] + _MAGS[c + 1])
        up = (m > mid) if c % 2 == 0 else (m >= mid)
        code = code + up.astype(np.int64)
    sign = np.signbit(q).astype(np.int64)
    return (sign << 3) | code


def shared_exponent(amax):
    """s = floor(log2(amax)) - E2M1_EMAX clamped to [-127, 127] (amax >= 0)."""
    amax = float(amax)
    if amax == 0.0:
        return -E8M0_BIAS
    # floor(log2(amax)) exactly, from the binary exponent (frexp: amax = f 2^e, f in [.5, 1))
    _, e = math.frexp(amax)
    s = (e - 1) - E2M1_EMAX
    return max(-E8M0_BIAS, min(E8M0_BIAS, s))


def mxfp4_quantize(x, K=None):
    """Quantize rows of x (float16 [rows, >= K]) along K.

    Returns (codes uint8 [rows, K], scales uint8 [rows, ceil(K / 32)]).
    """
    x = np.asarray(x)
    if x.dtype != np.float16:
        raise TypeError("the quantized operand is float16")
    if x.ndim != 2:
        raise ValueError("x must be 2-D")
    if K is None:
        K = x.shape[1]
    v = x[:, :K].astype(np.float64)
    rows = v.shape[0]
    nblk = (K + MX_BLOCK - 1) // MX_BLOCK
    codes = np.zeros((rows, K), dtype=np.uint8)
    scales = np.zeros((rows, nblk), dtype=np.uint8)
    for r in range(rows):
        for b in range(nblk):
            blk = v[r, b * MX_BLOCK:(b + 1) * MX_BLOCK]
            if not np.all(np.isfinite(blk)):
                scales[r, b] = E8M0_NAN
                continue  # codes stay 0
            s = shared_exponent(np.max(np.abs(blk)) if blk.size else 0.0)
            scales[r, b] = s + E8M0_BIAS
            codes[r, b * MX_BLOCK:(b + 1) * MX_BLOCK] = e2m1_round(np.ldexp(blk, -s))
    return codes, scales


def pack_e2m1(codes):
    """Codes [rows, K] -> bytes [rows, ceil(K / 2)]; byte p holds k = 2p in its
    low nibble and k = 2p + 1 in its high nibble (0 past K)."""
    codes = np.asarray(codes, dtype=np.uint8)
    rows, K = codes.shape
    padded = np.zeros((rows, K + (K & 1)), dtype=np.uint8)
    padded[:, :K] = codes
    return (padded[:, 0::2] | (padded[:, 1::2] << 4)).astype(np.uint8)


def mxfp4_dequantize(packed, scales, K):
    """Real values [rows, K] of packed MXFP4 rows: e2m1(code) * 2^(e - 127)."""
    codes = gemm_ref.unpack_e2m1(packed, K)
    scales = np.asarray(scales)
    nblk = (K + MX_BLOCK - 1) // MX_BLOCK
    if scales.shape[1] < nblk:
        raise ValueError("need %d scale bytes per row" % nblk)
    x = np.repeat(e8m0_decode(scales[:, :nblk]), MX_BLOCK, axis=1)[:, :K]
    return gemm_ref.e2m1_decode(codes) * x


def gemm_mx_reference(A, A_scales, B, B_scales, K, C=None, bias=None, alpha=1.0, beta=0.0,
                      epilogue="none", rows=None, program=None):
    """D_ref (float64) of D = epilogue(alpha * a.b^T + beta * C) for MXFP4 A
    (packed [M, >= K/2] + scales) and B (packed [N, >= K/2] + scales)."""
    A = np.asarray(A)
    A_scales = np.asarray(A_scales)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        A, A_scales = A[rows], A_scales[rows]
        if C is not None:
            C = np.asarray(C)[rows]
    a = mxfp4_dequantize(A, A_scales, K)
    b = mxfp4_dequantize(B, B_scales, K)
    return gemm_ref.fp_epilogue(a @ b.T, C, bias, alpha, beta, epilogue, program)


def error_bound_mx(A, A_scales, B, B_scales, K, D_ref, C=None, bias=None, alpha=1.0, beta=0.0,
                   epilogue="none", rows=None, program=None):
    """The FP16 path's acceptance bound (gemm_ref.error_bound) with the
    decoded MXFP4 operands in place of A and B."""
    A = np.asarray(A)
    A_scales = np.asarray(A_scales)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        A, A_scales = A[rows], A_scales[rows]
        if C is not None:
            C = np.asarray(C)[rows]
    a = mxfp4_dequantize(A, A_scales, K)
    b = mxfp4_dequantize(B, B_scales, K)
    return gemm_ref.fp_bound(a, b, D_ref, C, bias, alpha, beta, epilogue, program)
