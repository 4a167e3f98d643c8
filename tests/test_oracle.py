"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each check is a function of the GEMM definition under test, so the same checks
are also run against deliberately broken copies of the oracle (a transposed
operand, a dropped beta term, a flipped sign, swapped nibbles, a tanh GELU...)
to show that every such mistake fails at least one pin.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import gemm_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pairs(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


# ---------------------------------------------------------------------------
# E2M1 code table and packing
# ---------------------------------------------------------------------------

def _golden_e2m1():
    return {int(c): float(v) for c, v in _read_pairs("e2m1_codes.txt")}


def test_e2m1_table_matches_golden():
    table = _golden_e2m1()
    assert sorted(table) == list(range(16))
    for code, value in table.items():
        got = oracle.e2m1_value(code)
        assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value), code
    decoded = oracle.e2m1_decode(np.arange(16))
    assert np.array_equal(decoded, np.array([table[c] for c in range(16)]))


def test_e2m1_magnitudes_are_the_stated_set():
    mags = sorted({abs(oracle.e2m1_value(c)) for c in range(16)})
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_rejects_out_of_range():
    with pytest.raises(ValueError):
        oracle.e2m1_value(16)
    with pytest.raises(ValueError):
        oracle.e2m1_decode(np.array([3, 17]))


def _golden_pack():
    d = {r[0]: r[1:] for r in _read_pairs("e2m1_pack_vector.txt")}
    packed = np.array([[int(b, 16) for b in d["bytes"]]], dtype=np.uint8)
    codes = np.array([[int(c) for c in d["codes"]]])
    values = np.array([[float(v) for v in d["values"]]])
    return packed, codes, values


def test_unpack_matches_hand_built_vector():
    packed, codes, values = _golden_pack()
    K = codes.shape[1]
    got = oracle.unpack_e2m1(packed, K)
    assert np.array_equal(got, codes)
    assert np.array_equal(oracle.e2m1_decode(got), values)
    # odd K drops the last high nibble
    assert np.array_equal(oracle.unpack_e2m1(packed, K - 1), codes[:, : K - 1])


# ---------------------------------------------------------------------------
# GELU
# ---------------------------------------------------------------------------

def test_gelu_against_normal_cdf_table():
    for x, phi in _read_pairs("normal_cdf.txt"):
        x, phi = float(x), float(phi)
        assert abs(float(oracle.gelu_erf(x)) - x * phi) <= 1e-9 * max(1.0, abs(x))


def test_gelu_identities():
    xs = np.linspace(-8, 8, 161)
    g = oracle.gelu_erf(xs)
    assert oracle.gelu_erf(0.0) == 0.0
    assert np.allclose(g - oracle.gelu_erf(-xs), xs, rtol=0, atol=1e-12)  # GELU(x)-GELU(-x)=x
    big = xs[xs >= 6]
    assert np.all(np.abs(oracle.gelu_erf(big) - big) < 1e-7)
    # the Lipschitz constant used by the error bound really bounds GELU'
    fine = np.linspace(-10, 10, 200001)
    slope = np.abs(np.diff(oracle.gelu_erf(fine)) / np.diff(fine))
    assert slope.max() <= oracle.GELU_LIPSCHITZ
    assert slope.max() > 1.12


# ---------------------------------------------------------------------------
# The GEMM definition: checks written as functions of the definition
# ---------------------------------------------------------------------------

def _f16(x):
    return np.asarray(x, dtype=np.float16)


def check_identity(fn):
    rng = np.random.default_rng(1)
    M, K = 5, 7
    A = _f16(rng.uniform(-2, 2, (M, K)))
    eye = _f16(np.eye(K))                     # B as N=K rows of K
    D = fn(A, eye, K)
    return np.array_equal(D, A.astype(np.float64))


def check_permutation(fn):
    rng = np.random.default_rng(2)
    M, K = 4, 6
    A = _f16(rng.uniform(-2, 2, (M, K)))
    perm = np.array([3, 0, 5, 1, 4, 2])
    P = np.zeros((K, K), dtype=np.float16)
    P[np.arange(K), perm] = 1.0               # row j of B selects column perm[j] of A
    D = fn(A, P, K)
    return np.array_equal(D, A[:, perm].astype(np.float64))


def check_all_ones(fn):
    M, N, K = 3, 5, 256
    D = fn(_f16(np.ones((M, K))), _f16(np.ones((N, K))), K)
    return np.array_equal(D, np.full((M, N), float(K)))


def check_rank1(fn):
    # every row of A is u, every row of B is v  ->  D_ij = u . v for all i, j
    u = _f16([0.5, -1.25, 2.0, 0.125, -3.0, 1.0])
    v = _f16([4.0, 0.5, -0.25, 8.0, 1.5, -2.0])
    uv = 0.5 * 4.0 + -1.25 * 0.5 + 2.0 * -0.25 + 0.125 * 8.0 + -3.0 * 1.5 + 1.0 * -2.0  # = -4.625
    D = fn(np.tile(u, (3, 1)), np.tile(v, (4, 1)), 6)
    return np.array_equal(D, np.full((3, 4), -4.625)) and uv == -4.625


def check_rectangular_orientation(fn):
    # A 2x3, B given as N=4 rows of K=3; hand-computed D (2x4).
    A = _f16([[1, 2, 3], [-1, 0, 2]])
    B = _f16([[1, 0, 0], [0, 1, 0], [1, 1, 1], [2, -1, 0.5]])
    want = np.array([[1, 2, 6, 1.5], [-1, 0, 1, -1.0]])
    return np.array_equal(fn(A, B, 3), want)


def check_epilogue_alpha_beta_bias(fn):
    # A = 0: D = beta*C + bias exactly; alpha scales the product with its sign.
    M, N, K = 2, 3, 4
    C = _f16([[1, -2, 4], [0.5, 8, -16]])
    bias = _f16([0.25, -0.5, 1])
    D0 = fn(_f16(np.zeros((M, K))), _f16(np.ones((N, K))), K, C=C, bias=bias, alpha=3.0,
            beta=0.5, epilogue="bias")
    ok = np.array_equal(D0, np.array([[0.75, -1.5, 3.0], [0.5, 3.5, -7.0]]))
    D1 = fn(_f16(np.ones((M, K))), _f16(np.ones((N, K))), K, C=C, bias=bias, alpha=-2.0,
            beta=0.5, epilogue="bias")
    # -2*4 + 0.5*C + bias
    ok &= np.array_equal(D1, np.array([[-7.25, -9.5, -5.0], [-7.5, -4.5, -15.0]]))
    return bool(ok)


def check_gelu_after_bias(fn):
    # t = acc + bias with acc = 0 -> D = GELU(bias); 1 * Phi(1) from the table
    phi1 = 0.8413447461
    bias = _f16([1.0, -1.0])
    D = fn(_f16(np.zeros((1, 2))), _f16(np.zeros((2, 2))), 2, bias=bias, epilogue="bias_gelu")
    return abs(D[0, 0] - phi1) < 1e-9 and abs(D[0, 1] - (-1.0) * (1 - phi1)) < 1e-9


def check_int8_extremes(fn):
    K = 4096
    A = np.full((2, K), -128, dtype=np.int8)
    D = fn(A, np.full((3, K), -128, dtype=np.int8), K, "i8", "i8")
    ok = np.array_equal(D, np.full((2, 3), K * 16384))          # 2^26
    D2 = fn(np.full((1, K), 127, dtype=np.int8), np.full((2, K), -128, dtype=np.int8), K,
            "i8", "i8")
    ok &= np.array_equal(D2, np.full((1, 2), -K * 16256))
    return bool(ok)


def check_int8_wrap(fn):
    # A = B = 127, K = 16: acc = 16 * 16129 = 258064; alpha = 65536:
    # 258064 * 65536 = 16912482304 = 3 * 2^32 + 4027580416 -> int32 -267386880.
    K = 16
    D = fn(np.full((1, K), 127, dtype=np.int8), np.full((1, K), 127, dtype=np.int8), K,
           "i8", "i8", alpha=65536)
    # beta * C with C = -7, beta = 3, alpha = 1: acc - 21
    C = np.full((1, 1), -7, dtype=np.int32)
    D2 = fn(np.full((1, K), 127, dtype=np.int8), np.full((1, K), 127, dtype=np.int8), K,
            "i8", "i8", C=C, alpha=1, beta=3)
    return int(D[0, 0]) == -267386880 and int(D2[0, 0]) == 258064 - 21


def check_e2m1_one_hot(fn):
    # weight column j has one nonzero code c_j at k_j: D[:, j] = A[:, k_j] * value(c_j)
    table = _golden_e2m1()
    K, N = 8, 16
    rng = np.random.default_rng(3)
    A = _f16(rng.uniform(-4, 4, (3, K)))
    packed = np.zeros((N, K // 2), dtype=np.uint8)
    ks = [(3 * j + 1) % K for j in range(N)]
    for j in range(N):
        k = ks[j]
        packed[j, k // 2] |= np.uint8(j << (4 * (k % 2)))       # code j
    D = fn(A, packed, K, "f16", "e2m1")
    want = np.stack([A[:, ks[j]].astype(np.float64) * table[j] for j in range(N)], axis=1)
    return np.array_equal(D, want)


def _exact_e2m1(packed_row, k, table):
    byte = int(packed_row[k // 2])
    code = (byte >> 4) if (k % 2) else (byte & 15)
    return Fraction(table[code])


def _brute(A, B, K, dtype_a, dtype_b, C, bias, alpha, beta, epilogue):
    """Exact rational GEMM with pure-Python loops (tiny shapes only)."""
    table = _golden_e2m1()
    M = A.shape[0]
    N = B.shape[0]
    out = [[None] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            for k in range(K):
                a = Fraction(int(A[i, k])) if dtype_a == "i8" else Fraction(float(A[i, k]))
                if dtype_b == "e2m1":
                    b = _exact_e2m1(B[j], k, table)
                elif dtype_b == "i8":
                    b = Fraction(int(B[j, k]))
                else:
                    b = Fraction(float(B[j, k]))
                s += a * b
            t = Fraction(alpha) * s
            if beta:
                cval = int(C[i, j]) if dtype_a == "i8" else float(C[i, j])
                t += Fraction(beta) * Fraction(cval)
            if bias is not None:
                t += Fraction(float(bias[j]))
            out[i][j] = t
    return out


def check_brute_force(fn, seed=0):
    """Random tiny shapes against exact rational arithmetic."""
    rng = np.random.default_rng(100 + seed)
    ok = True
    for trial in range(12):
        M, N, K = (int(x) for x in rng.integers(1, 9, size=3))
        pair = [("f16", "f16"), ("i8", "i8"), ("f16", "e2m1")][trial % 3]
        epi = ["none", "bias", "gelu", "bias_gelu"][trial % 4] if pair[0] == "f16" else "none"
        if pair[0] == "i8":
            A = rng.integers(-128, 128, (M, K)).astype(np.int8)
            B = rng.integers(-128, 128, (N, K)).astype(np.int8)
            C = rng.integers(-1000, 1000, (M, N)).astype(np.int32)
            alpha, beta = int(rng.integers(-3, 4)), int(rng.integers(-2, 3))
        else:
            A = _f16(rng.standard_normal((M, K)))
            if pair[1] == "e2m1":
                B = rng.integers(0, 256, (N, (K + 1) // 2)).astype(np.uint8)
            else:
                B = _f16(rng.standard_normal((N, K)))
            C = _f16(rng.standard_normal((M, N)))
            alpha, beta = float(rng.choice([1.0, -0.75, 2.5])), float(rng.choice([0.0, 0.5, -1.25]))
        bias = _f16(rng.standard_normal(N)) if epi in ("bias", "bias_gelu") else None
        D = fn(A, B, K, pair[0], pair[1], C=C if beta else None, bias=bias, alpha=alpha,
               beta=beta, epilogue=epi)
        exact = _brute(A, B, K, pair[0], pair[1], C, bias, alpha, beta, epi)
        for i in range(M):
            for j in range(N):
                t = exact[i][j]
                if pair[0] == "i8":
                    want = ((int(t) + (1 << 31)) % (1 << 32)) - (1 << 31)
                    ok &= int(D[i, j]) == want
                    continue
                if epi in ("gelu", "bias_gelu"):
                    tf = float(t)
                    want = 0.5 * tf * (1.0 + math.erf(tf / math.sqrt(2.0)))
                    ok &= abs(D[i, j] - want) <= 1e-12 * max(1.0, abs(want))
                else:
                    ok &= abs(Fraction(float(D[i, j])) - t) <= abs(t) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 60)
    return bool(ok)


def check_rows_subset(fn):
    rng = np.random.default_rng(5)
    A = _f16(rng.standard_normal((9, 13)))
    B = _f16(rng.standard_normal((7, 13)))
    C = _f16(rng.standard_normal((9, 7)))
    full = fn(A, B, 13, C=C, beta=0.5)
    rows = np.array([8, 0, 3])
    part = fn(A, B, 13, C=C, beta=0.5, rows=rows)
    return np.array_equal(part, full[rows])


# Epilogue programs.  acc = [-3, 0.5, 2, 7] from a K = 1 product; every
# expected row below is worked out by hand from the op definitions (t + b_j,
# max(t, 0), GELU(t) = t Phi(t), a t, min(max(t, lo), hi)), applied in order.
_PROG_A = _f16([[1.0]])
_PROG_B = _f16([[-3.0], [0.5], [2.0], [7.0]])
_PROG_BIAS = _f16([1.0, -1.0, 0.5, -8.0])
_PROG_CASES = [
    ([], 1.0, [-3.0, 0.5, 2.0, 7.0]),
    (["relu"], 1.0, [0.0, 0.5, 2.0, 7.0]),
    ([("scale", -0.5)], 1.0, [1.5, -0.25, -1.0, -3.5]),
    ([("clamp", -1.0, 2.5)], 1.0, [-1.0, 0.5, 2.0, 2.5]),
    (["relu", ("scale", -1.0)], 1.0, [0.0, -0.5, -2.0, -7.0]),
    ([("scale", -1.0), "relu"], 1.0, [3.0, 0.0, 0.0, 0.0]),
    (["bias", "relu"], 1.0, [0.0, 0.0, 2.5, 0.0]),
    (["relu", "bias"], 1.0, [1.0, -0.5, 2.5, -1.0]),
    (["relu", ("clamp", 0.25, 1.0), ("scale", 4.0)], 2.0, [1.0, 4.0, 4.0, 4.0]),
    # int8 output: round half to even, then saturate
    ([("quant_i8", 2.0)], 1.0, [-6.0, 1.0, 4.0, 14.0]),
    ([("quant_i8", 0.25)], 1.0, [-1.0, 0.0, 0.0, 2.0]),     # -0.75, 0.125, 0.5, 1.75
    ([("quant_i8", 0.75)], 1.0, [-2.0, 0.0, 2.0, 5.0]),     # -2.25, 0.375, 1.5, 5.25
    ([("scale", 100.0), ("quant_i8", 1.0)], 1.0, [-128.0, 50.0, 127.0, 127.0]),
    (["bias", ("quant_i8", -1.0)], 1.0, [2.0, 0.0, -2.0, 1.0]),   # -(t + bias) = 2, .5, -2.5, 1
]


def check_program_by_hand(fn):
    for prog, alpha, want in _PROG_CASES:
        got = fn(_PROG_A, _PROG_B, 1, bias=_PROG_BIAS, alpha=alpha, program=prog)
        if not np.array_equal(got, np.array([want])):
            return False
    return True


def check_program_after_alpha_beta(fn):
    # t = 2 acc - C = [-7, 0, 3, 13], then clamp to [-5, 5]
    C = _f16([[1.0, 1.0, 1.0, 1.0]])
    got = fn(_PROG_A, _PROG_B, 1, C=C, alpha=2.0, beta=-1.0, program=[("clamp", -5.0, 5.0)])
    return np.array_equal(got, np.array([[-5.0, 0.0, 3.0, 5.0]]))


def check_program_gelu_table(fn):
    # GELU(x) = x Phi(x) with Phi from the printed normal-CDF table (10 digits),
    # after a bias op that moves acc = [-3, 0.5, 2, 7] to [-2, -0.5, 2.5, -1]
    phi = {float(x): float(p) for x, p in _read_pairs("normal_cdf.txt")}
    got = fn(_PROG_A, _PROG_B, 1, bias=_PROG_BIAS, program=["bias", "gelu"])
    want = [-2.0 * phi[-2.0], -0.5 * (1.0 - phi[0.5]), 2.5 * phi[2.5], -1.0 * phi[-1.0]]
    return np.allclose(got, np.array([want]), rtol=0, atol=1e-9)


def check_program_operands_are_binary32(fn):
    # 0.1 is passed as the binary32 number 13421773 / 2^27, not the decimal 0.1
    got = fn(_PROG_A, _f16([[1.0]]), 1, program=[("scale", 0.1)])
    return got[0, 0] == 13421773 / 2.0 ** 27


ALL_CHECKS = [check_identity, check_permutation, check_all_ones, check_rank1,
              check_rectangular_orientation, check_epilogue_alpha_beta_bias,
              check_gelu_after_bias, check_int8_extremes, check_int8_wrap,
              check_e2m1_one_hot, check_brute_force, check_rows_subset,
              check_program_by_hand, check_program_after_alpha_beta, check_program_gelu_table,
              check_program_operands_are_binary32]


def _ref(A, B, K, dtype_a="f16", dtype_b="f16", **kw):
    return oracle.gemm_reference(A, B, K, dtype_a, dtype_b, **kw)


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    assert check(_ref)


# ---------------------------------------------------------------------------
# Planted mistakes: each broken copy of the oracle must fail some pin.
# ---------------------------------------------------------------------------

def _mutant(patch):
    def fn(A, B, K, dtype_a="f16", dtype_b="f16", **kw):
        with patch():
            return oracle.gemm_reference(A, B, K, dtype_a, dtype_b, **kw)
    return fn


class _Swap:
    def __init__(self, name, new):
        self.name, self.new = name, new

    def __call__(self):
        return self

    def __enter__(self):
        self.old = getattr(gemm_ref, self.name)
        setattr(gemm_ref, self.name, self.new)

    def __exit__(self, *a):
        setattr(gemm_ref, self.name, self.old)


def _mut_transpose_b(B, dtype_b, K):
    b = _ORIG_OPERAND_B(B, dtype_b, K)
    return b.T if b.shape[0] == b.shape[1] else b[::-1]


def _mut_nibbles(packed, K):
    packed = np.asarray(packed, dtype=np.uint8)
    swapped = ((packed & 0x0F) << 4) | (packed >> 4)
    return _ORIG_UNPACK(swapped.astype(np.uint8), K)


def _mut_tanh_gelu(t):
    t = np.asarray(t, dtype=np.float64)
    return 0.5 * t * (1 + np.tanh(math.sqrt(2 / math.pi) * (t + 0.044715 * t ** 3)))


def _mut_decode_bias0(codes):
    codes = np.asarray(codes).astype(np.int64)
    s = np.where(codes & 8, -1.0, 1.0)
    e = (codes >> 1) & 3
    m = codes & 1
    return s * np.where(e == 0, 0.5 * m, 2.0 ** e * (1 + 0.5 * m))  # exponent bias 0


def _mut_drop_sign(codes):
    return np.abs(_ORIG_DECODE(codes))


def _mut_operand_a_abs(A, dtype_a):
    return np.abs(_ORIG_OPERAND_A(A, dtype_a))


def _mut_wrap_saturate(x_u64):
    v = x_u64.astype(np.int64)
    return np.clip(v, -(1 << 31), (1 << 31) - 1)


_ORIG_OPERAND_B = gemm_ref._operand_b
_ORIG_OPERAND_A = gemm_ref._operand_a
_ORIG_UNPACK = gemm_ref.unpack_e2m1
_ORIG_DECODE = gemm_ref.e2m1_decode


class _DropBeta:
    """Plants 'beta*C forgotten' by zeroing beta on the way in."""

    def __call__(self):
        return self

    def __enter__(self):
        self.old = gemm_ref.gemm_reference
        old = self.old

        def patched(*a, **kw):
            kw["beta"] = 0.0
            return old(*a, **kw)
        oracle.gemm_reference = patched

    def __exit__(self, *a):
        oracle.gemm_reference = self.old


class _BiasBeforeAlpha:
    """Plants 'bias scaled by alpha' (wrong epilogue order)."""

    def __call__(self):
        return self

    def __enter__(self):
        self.old = gemm_ref.gemm_reference
        old = self.old

        def patched(A, B, K, dtype_a="f16", dtype_b="f16", C=None, bias=None, alpha=1.0,
                    beta=0.0, epilogue="none", rows=None, program=None):
            if bias is not None and (epilogue in ("bias", "bias_gelu") or program):
                bias = (np.asarray(bias, dtype=np.float64) * alpha).astype(np.float16)
            return old(A, B, K, dtype_a, dtype_b, C=C, bias=bias, alpha=alpha, beta=beta,
                       epilogue=epilogue, rows=rows, program=program)
        oracle.gemm_reference = patched

    def __exit__(self, *a):
        oracle.gemm_reference = self.old


_ORIG_APPLY_PROGRAM = gemm_ref.apply_program


def _mut_program_reversed(t, program, bias=None):
    return _ORIG_APPLY_PROGRAM(t, list(program)[::-1], bias)


def _mut_relu_abs(t, program, bias=None):
    for op in program:
        if op == "relu" or (isinstance(op, tuple) and op[0] == "relu"):
            t = np.abs(np.asarray(t, dtype=np.float64))
        else:
            t = _ORIG_APPLY_PROGRAM(t, [op], bias)
    return t


def _mut_clamp_order(t, program, bias=None):
    # the bounds swapped: max(min(t, lo), hi)
    for op in program:
        if isinstance(op, tuple) and op[0] == "clamp":
            t = np.maximum(np.minimum(t, op[1]), op[2])
        else:
            t = _ORIG_APPLY_PROGRAM(t, [op], bias)
    return t


def _mut_round_half_up(t, program, bias=None):
    # quantization rounding half away from zero instead of half to even
    for op in program:
        if isinstance(op, tuple) and op[0] == "quant_i8":
            x = float(np.float32(op[1])) * np.asarray(t, dtype=np.float64)
            t = np.clip(np.sign(x) * np.floor(np.abs(x) + 0.5), -128, 127)
        else:
            t = _ORIG_APPLY_PROGRAM(t, [op], bias)
    return t


def _mut_wrap_i8(t, program, bias=None):
    # quantization wrapping modulo 256 instead of saturating
    for op in program:
        if isinstance(op, tuple) and op[0] == "quant_i8":
            x = np.rint(float(np.float32(op[1])) * np.asarray(t, dtype=np.float64))
            t = ((x + 128) % 256) - 128
        else:
            t = _ORIG_APPLY_PROGRAM(t, [op], bias)
    return t


def _mut_scale_decimal(t, program, bias=None):
    # scale operand kept as the decimal (binary64) value, not binary32
    for op in program:
        if isinstance(op, tuple) and op[0] == "scale":
            t = op[1] * np.asarray(t, dtype=np.float64)
        else:
            t = _ORIG_APPLY_PROGRAM(t, [op], bias)
    return t


MUTANTS = {
    "program_reversed": _Swap("apply_program", _mut_program_reversed),
    "relu_as_abs": _Swap("apply_program", _mut_relu_abs),
    "clamp_order": _Swap("apply_program", _mut_clamp_order),
    "scale_binary64": _Swap("apply_program", _mut_scale_decimal),
    "quant_round_half_up": _Swap("apply_program", _mut_round_half_up),
    "quant_wraps": _Swap("apply_program", _mut_wrap_i8),
    "transposed_B": _Swap("_operand_b", _mut_transpose_b),
    "swapped_nibbles": _Swap("unpack_e2m1", _mut_nibbles),
    "tanh_gelu": _Swap("gelu_erf", _mut_tanh_gelu),
    "e2m1_bias0": _Swap("e2m1_decode", _mut_decode_bias0),
    "e2m1_no_sign": _Swap("e2m1_decode", _mut_drop_sign),
    "abs_A": _Swap("_operand_a", _mut_operand_a_abs),
    "int8_saturates": _Swap("_wrap_int32", _mut_wrap_saturate),
    "dropped_beta": _DropBeta(),
    "bias_times_alpha": _BiasBeforeAlpha(),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name):
    fn = _mutant(MUTANTS[name])
    failed = []
    for check in ALL_CHECKS:
        try:
            ok = check(fn)
        except Exception:
            ok = False
        if not ok:
            failed.append(check.__name__)
    assert failed, "mutant %s passed every pin" % name


# ---------------------------------------------------------------------------
# The acceptance bound
# ---------------------------------------------------------------------------

def test_error_bound_terms():
    A = _f16([[1.0, -2.0]])
    B = _f16([[3.0, 0.5], [-1.0, -1.0]])
    C = _f16([[4.0, -8.0]])
    bias = _f16([0.5, -0.25])
    D = oracle.gemm_reference(A, B, 2, C=C, bias=bias, alpha=2.0, beta=-0.5, epilogue="bias")
    # acc = [2, 1]; t = 2*acc - 0.5*C + bias = [2.5, 5.75]
    assert np.array_equal(D, np.array([[2.5, 5.75]]))
    bnd = oracle.error_bound(A, B, 2, D, C=C, bias=bias, alpha=2.0, beta=-0.5, epilogue="bias")
    # P = 2*(|A|.|B|) + 0.5|C| + |bias| = [2*4+2+0.5, 2*3+4+0.25] = [10.5, 10.25]
    want = 2.0 ** -10 * np.array([[10.5, 10.25]]) + 2.0 ** -10 * np.array([[2.5, 5.75]]) + 2.0 ** -24
    assert np.array_equal(bnd, want)
    Dg = oracle.gemm_reference(A, B, 2, C=C, bias=bias, alpha=2.0, beta=-0.5, epilogue="bias_gelu")
    bg = oracle.error_bound(A, B, 2, Dg, C=C, bias=bias, alpha=2.0, beta=-0.5, epilogue="bias_gelu")
    assert np.allclose(bg, oracle.GELU_LIPSCHITZ * 2.0 ** -10 * np.array([[10.5, 10.25]])
                       + 2.0 ** -10 * np.abs(Dg) + 2.0 ** -24, rtol=1e-15, atol=0)


def test_fp16_rounding_fits_in_bound():
    # Rounding D_ref to fp16 (round-to-nearest-even) must always pass the bound,
    # including fp16 subnormals and values near the fp16 maximum.
    rng = np.random.default_rng(7)
    vals = np.concatenate([rng.standard_normal(10000) * 10.0 ** rng.integers(-8, 4, 10000),
                           [0.0, 2.0 ** -24, 3 * 2.0 ** -25, 65000.0]])
    rounded = vals.astype(np.float16).astype(np.float64)
    bound = 2.0 ** -10 * np.abs(vals) + 2.0 ** -24
    assert np.all(np.abs(rounded - vals) <= bound)


def test_error_bound_program_terms():
    # acc = [2, 1], t = 2 acc = [4, 2], P_0 = 2 (|A|.|B|) = [8, 6]
    A = _f16([[1.0, -2.0]])
    B = _f16([[3.0, 0.5], [-1.0, -1.0]])
    prog = [("scale", -0.5), "relu", "gelu"]
    D = oracle.gemm_reference(A, B, 2, alpha=2.0, program=prog)
    assert np.array_equal(D, np.array([[0.0, 0.0]]))  # scale -> [-2, -1], relu -> 0, GELU(0) = 0
    bnd = oracle.error_bound(A, B, 2, D, alpha=2.0, program=prog)
    # scale: 0.5 * 2^-10 [8, 6] + 2^-20 [2, 1]; relu: + 0; GELU: * 1.13, + 0
    want = 1.13 * (2.0 ** -10 * np.array([[4.0, 3.0]]) + 2.0 ** -20 * np.array([[2.0, 1.0]]))
    assert np.allclose(bnd, want + 2.0 ** -24, rtol=1e-15, atol=0)
    bias = _f16([0.5, -4.0])
    prog = ["bias", ("clamp", -1.0, 1.0)]
    D = oracle.gemm_reference(A, B, 2, bias=bias, alpha=2.0, program=prog)
    assert np.array_equal(D, np.array([[1.0, -1.0]]))  # t + bias = [4.5, -2]
    bnd = oracle.error_bound(A, B, 2, D, bias=bias, alpha=2.0, program=prog)
    want = (2.0 ** -10 * np.array([[8.5, 10.0]]) + 2.0 ** -20 * np.array([[4.5, 2.0]])
            + 2.0 ** -20 * np.array([[1.0, 1.0]]) + 2.0 ** -10 * np.array([[1.0, 1.0]]) + 2.0 ** -24)
    assert np.allclose(bnd, want, rtol=1e-15, atol=0)


def test_error_bound_quant_terms():
    # t = 2 acc = [4, 2], E = 2^-10 [8, 6]; quant a = 3: |a| E + 1, then no
    # per-op rounding term; D = [12, 6]
    A = _f16([[1.0, -2.0]])
    B = _f16([[3.0, 0.5], [-1.0, -1.0]])
    prog = [("quant_i8", 3.0)]
    D = oracle.gemm_reference(A, B, 2, alpha=2.0, program=prog)
    assert np.array_equal(D, np.array([[12.0, 6.0]]))
    bnd = oracle.error_bound(A, B, 2, D, alpha=2.0, program=prog)
    want = 3.0 * 2.0 ** -10 * np.array([[8.0, 6.0]]) + 1.0 + 2.0 ** -10 * np.array([[12.0, 6.0]])
    assert np.allclose(bnd, want + 2.0 ** -24, rtol=1e-15, atol=0)


def test_quantize_special_values():
    q = oracle.quantize_i8(np.array([np.nan, np.inf, -np.inf, 127.5, -128.5, 2.5, -2.5, 0.49999]))
    assert q.tolist() == [0.0, 127.0, -128.0, 127.0, -128.0, 2.0, -2.0, 0.0]


def test_program_rejects_bad_ops():
    A, B = _PROG_A, _PROG_B
    for prog in (["tanh"], [("scale",)], [("clamp", 2.0, 1.0)], [("relu", 1.0)],
                 [("quant_i8", 1.0), "relu"]):
        with pytest.raises(ValueError):
            oracle.gemm_reference(A, B, 1, program=prog)
    with pytest.raises(ValueError):
        oracle.gemm_reference(A, B, 1, program=["bias"])  # no bias vector
    with pytest.raises(ValueError):
        oracle.gemm_reference(A, B, 1, epilogue="gelu", program=["relu"])
