"""Pins of the MXFP4 oracle (oracle.mx_ref) against facts that do not come
from the oracle itself: the E8M0 format's values, a brute-force search for the
nearest E2M1 value, the characterisation of the block scale (amax / X lies in
[4, 8) for every non-zero block), blocks already on the grid, special blocks,
and exact rational sums for the GEMM.  Each check also runs against broken
copies of the oracle, every one of which must fail some check."""

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import gemm_ref, mx_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # E2M1 magnitudes, by hand


def _golden_e8m0():
    out = {}
    with open(os.path.join(GOLDEN, "e8m0_values.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                c, v = line.split()
                out[int(c)] = float(v)
    return out


def _brute_round(q):
    """Nearest of the eight magnitudes by exhaustive search; at equal
    distance the even code (mantissa bit 0) wins; sign bit from q."""
    m = abs(q)
    best = min(range(8), key=lambda c: (abs(m - MAGS[c]), c % 2))
    return best | (8 if math.copysign(1.0, q) < 0 else 0)


# ---------------------------------------------------------------------------
# Checks: each takes nothing and reads the oracle through the module, so that
# a planted mistake (an attribute swapped on the module) is seen.
# ---------------------------------------------------------------------------

def check_e8m0_golden():
    g = _golden_e8m0()
    for c, v in g.items():
        got = mx_ref.e8m0_value(c)
        if math.isnan(v) != math.isnan(got) or (not math.isnan(v) and got != v):
            return False
    return True


def check_rounding_brute_force():
    rng = np.random.default_rng(1)
    q = list(rng.uniform(-9, 9, 4000))
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    for m in mids + MAGS + [6.5, 7.0, 7.99, 100.0]:
        for s in (1.0, -1.0):
            q += [s * m, s * np.nextafter(m, 0), s * np.nextafter(m, 10)]
    q += [0.0, -0.0]
    got = mx_ref.e2m1_round(np.array(q))
    return all(int(g) == _brute_round(x) for g, x in zip(got, q))


def check_rounding_by_hand():
    # hand-worked: ties to the even mantissa bit, saturation, kept signs
    cases = [(0.25, 0), (0.26, 1), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6),
             (5.0, 6), (5.01, 7), (6.0, 7), (7.9, 7), (100.0, 7), (-0.25, 8), (-0.0, 8),
             (0.0, 0), (-5.5, 15), (-1.0, 10)]
    got = mx_ref.e2m1_round(np.array([q for q, _ in cases]))
    return [int(g) for g in got] == [c for _, c in cases]


def _block(values, K=32):
    x = np.zeros((1, K), dtype=np.float16)
    x[0, :len(values)] = values
    return x


def check_scale_of_powers_of_two():
    # amax = 2^p exactly: X = 2^(p-2), amax/X = 4, code 6 (value 4)
    for p in range(-24, 16):
        codes, scales = mx_ref.mxfp4_quantize(_block([2.0 ** p]))
        if scales[0, 0] != p - 2 + 127 or codes[0, 0] != 6:
            return False
    # amax just below 2^p: X = 2^(p-3), amax/X just below 8, saturated to 6
    for p in range(-10, 16):
        v = np.float16(2.0 ** p) - np.float16(2.0 ** (p - 11))
        codes, scales = mx_ref.mxfp4_quantize(_block([v]))
        if scales[0, 0] != p - 3 + 127 or codes[0, 0] != 7:
            return False
    return True


def check_scale_characterisation():
    # for every non-zero finite block: amax / X in [4, 8), X = 2^(e - 127)
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((16, 256)) * np.exp2(rng.integers(-20, 12, (16, 1)))).astype(np.float16)
    codes, scales = mx_ref.mxfp4_quantize(x)
    if scales.shape != (16, 8):
        return False
    for r in range(16):
        for b in range(8):
            amax = float(np.max(np.abs(x[r, 32 * b:32 * b + 32].astype(np.float64))))
            ratio = amax / math.ldexp(1.0, int(scales[r, b]) - 127)
            if not 4.0 <= ratio < 8.0:
                return False
    return True


def check_error_within_half_spacing():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((8, 128)) * 3).astype(np.float16)
    codes, scales = mx_ref.mxfp4_quantize(x)
    deq = mx_ref.mxfp4_dequantize(mx_ref.pack_e2m1(codes), scales, 128)
    X = np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)
    m = np.abs(x.astype(np.float64)) / X
    spacing = np.where(m < 2, 0.5, np.where(m < 4, 1.0, 2.0))
    err = np.abs(deq - x.astype(np.float64)) / X
    ok = np.where(m <= 6, err <= spacing / 2, err < 2.0)
    return bool(ok.all()) and np.array_equal(np.signbit(deq), np.signbit(x.astype(np.float64)))


def check_grid_blocks_reconstruct():
    # values already of the form e2m1 * 2^s, with a code of magnitude 4 or 6
    # in the block, come back unchanged, scale s + 127
    rng = np.random.default_rng(4)
    for s in (-23, -10, -1, 0, 3, 13):
        c = rng.integers(0, 16, 64)
        c[5], c[40] = 7, 14
        vals = np.array([math.ldexp(MAGS[k & 7] * (-1 if k & 8 else 1), s) for k in c])
        x = vals.astype(np.float16)[None, :]
        assert np.array_equal(x.astype(np.float64)[0], vals)
        codes, scales = mx_ref.mxfp4_quantize(x)
        if not (np.array_equal(codes[0], c) and list(scales[0]) == [s + 127, s + 127]):
            return False
        deq = mx_ref.mxfp4_dequantize(mx_ref.pack_e2m1(codes), scales, 64)
        if not np.array_equal(deq[0], vals):
            return False
    return True


def check_special_blocks():
    x = np.ones((1, 128), dtype=np.float16)
    x[0, 3] = np.nan
    x[0, 40] = np.inf
    x[0, 64:96] = 0.0
    x[0, 96:128] = -0.0
    codes, scales = mx_ref.mxfp4_quantize(x)
    return (list(scales[0]) == [255, 255, 0, 0] and not codes[0, :64].any()
            and not codes[0, 64:96].any() and (codes[0, 96:] == 8).all())


def check_ragged_last_block():
    # K = 40: blocks of 32 and 8 values, each with its own scale
    x = np.full((2, 40), 0.001, dtype=np.float16)
    x[0, 35] = 100.0    # large value in the short block only
    x[1, 3] = 100.0     # large value in the full block only
    codes, scales = mx_ref.mxfp4_quantize(x)
    # 100 = 1.5625 * 2^6: X = 2^4; 0.001 ~ 2^-9.97: X = 2^-12
    return (scales.shape == (2, 2) and list(scales[0]) == [115, 131]
            and list(scales[1]) == [131, 115])


def check_pack_layout():
    packed = mx_ref.pack_e2m1(np.array([[1, 2, 3]], dtype=np.uint8))
    return (packed.tolist() == [[0x21, 0x03]]
            and np.array_equal(gemm_ref.unpack_e2m1(packed, 3), [[1, 2, 3]]))


def _exact_gemm(Ac, As, Bc, Bs, K):
    """Exact rational product of decoded MXFP4 operands (codes unpacked)."""
    def val(c, s):
        m = Fraction(MAGS[c & 7]).limit_denominator() * (-1 if c & 8 else 1)
        return m * (Fraction(2) ** (int(s) - 127))
    M, N = len(Ac), len(Bc)
    out = [[Fraction(0)] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            out[i][j] = sum(val(Ac[i][k], As[i][k // 32]) * val(Bc[j][k], Bs[j][k // 32])
                            for k in range(K))
    return out


def check_gemm_brute_force():
    rng = np.random.default_rng(5)
    for (M, N, K) in [(1, 1, 1), (2, 3, 33), (3, 2, 70), (1, 4, 64)]:
        nb = (K + 31) // 32
        Ac = rng.integers(0, 16, (M, K)).astype(np.uint8)
        Bc = rng.integers(0, 16, (N, K)).astype(np.uint8)
        As = rng.integers(110, 140, (M, nb)).astype(np.uint8)
        Bs = rng.integers(110, 140, (N, nb)).astype(np.uint8)
        D = mx_ref.gemm_mx_reference(mx_ref.pack_e2m1(Ac), As, mx_ref.pack_e2m1(Bc), Bs, K)
        ex = _exact_gemm(Ac.tolist(), As.tolist(), Bc.tolist(), Bs.tolist(), K)
        for i in range(M):
            for j in range(N):
                if abs(Fraction(float(D[i, j])) - ex[i][j]) > abs(ex[i][j]) * Fraction(1, 2 ** 50):
                    return False
    return True


def check_gemm_closed_form():
    # every code 1.0 (code 2): D_ij = sum over blocks of (values in block) *
    # 2^(sa + sb - 254); K = 80 has blocks of 32, 32, 16
    K = 80
    A = mx_ref.pack_e2m1(np.full((2, K), 2, dtype=np.uint8))
    B = mx_ref.pack_e2m1(np.full((3, K), 2, dtype=np.uint8))
    As = np.array([[127, 128, 120], [100, 127, 130]], dtype=np.uint8)
    Bs = np.array([[127, 127, 127], [126, 129, 131], [140, 110, 127]], dtype=np.uint8)
    D = mx_ref.gemm_mx_reference(A, As, B, Bs, K, C=np.ones((2, 3), np.float16), beta=0.5,
                                 alpha=2.0)
    n = [32, 32, 16]
    for i in range(2):
        for j in range(3):
            want = 2.0 * sum(n[b] * 2.0 ** (int(As[i, b]) + int(Bs[j, b]) - 254)
                             for b in range(3)) + 0.5
            if D[i, j] != want:
                return False
    return True


ALL_CHECKS = [check_e8m0_golden, check_rounding_brute_force, check_rounding_by_hand,
              check_scale_of_powers_of_two, check_scale_characterisation,
              check_error_within_half_spacing, check_grid_blocks_reconstruct,
              check_special_blocks, check_ragged_last_block, check_pack_layout,
              check_gemm_brute_force, check_gemm_closed_form]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    assert check()


# ---------------------------------------------------------------------------
# Planted mistakes
# ---------------------------------------------------------------------------

_ORIG = {n: getattr(mx_ref, n) for n in ("e2m1_round", "shared_exponent", "mxfp4_quantize",
                                          "e8m0_value", "mxfp4_dequantize", "pack_e2m1")}
_ORIG_CONST = {"E2M1_EMAX": mx_ref.E2M1_EMAX, "MX_BLOCK": mx_ref.MX_BLOCK}


def _round_ties_away(q):
    q = np.asarray(q, dtype=np.float64)
    m = np.abs(q)
    code = np.zeros(m.shape, dtype=np.int64)
    for c in range(7):
        code = code + (m >= 0.5 * (MAGS[c] + MAGS[c + 1])).astype(np.int64)
    return (np.signbit(q).astype(np.int64) << 3) | code


def _round_no_saturation(q):
    # values past 7 round to "8", which lands in the sign bit
    out = _ORIG["e2m1_round"](q)
    big = np.abs(np.asarray(q, dtype=np.float64)) >= 7.0
    return np.where(big, (out & 8) + 8, out) & 15


def _round_drop_sign(q):
    return _ORIG["e2m1_round"](np.abs(np.asarray(q, dtype=np.float64)))


def _shared_ceil(amax):
    if amax == 0:
        return -127
    return max(-127, min(127, math.ceil(math.log2(amax)) - 2))


def _quantize_row_scale(x, K=None):
    # one scale for the whole row instead of one per block
    x = np.asarray(x)
    K = x.shape[1] if K is None else K
    codes, scales = _ORIG["mxfp4_quantize"](x, K)
    v = x[:, :K].astype(np.float64)
    for r in range(v.shape[0]):
        if not np.all(np.isfinite(v[r])):
            continue
        s = _ORIG["shared_exponent"](float(np.max(np.abs(v[r]))))
        scales[r, :] = s + 127
        codes[r] = mx_ref.e2m1_round(np.ldexp(v[r], -s))
    return codes, scales


def _e8m0_bias_128(code):
    return float("nan") if code == 255 else math.ldexp(1.0, int(code) - 128)


class _Swap:
    def __init__(self, name, new):
        self.name, self.new = name, new

    def __enter__(self):
        self.old = getattr(mx_ref, self.name)
        setattr(mx_ref, self.name, self.new)

    def __exit__(self, *a):
        setattr(mx_ref, self.name, self.old)


MUTANTS = {
    "emax_3": _Swap("E2M1_EMAX", 3),
    "block_16": _Swap("MX_BLOCK", 16),
    "ceil_log2": _Swap("shared_exponent", _shared_ceil),
    "ties_away": _Swap("e2m1_round", _round_ties_away),
    "no_saturation": _Swap("e2m1_round", _round_no_saturation),
    "sign_lost": _Swap("e2m1_round", _round_drop_sign),
    "row_scale": _Swap("mxfp4_quantize", _quantize_row_scale),
    "e8m0_bias_128": _Swap("e8m0_value", _e8m0_bias_128),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name):
    failed = []
    with MUTANTS[name]:
        for check in ALL_CHECKS:
            try:
                ok = check()
            except Exception:
                ok = False
            if not ok:
                failed.append(check.__name__)
    assert failed, "mutant %s passed every pin" % name


def test_error_bound_mx_is_the_fp16_bound_on_decoded_operands():
    # with operands that are exactly FP16 values, the MXFP4 bound equals the
    # FP16 path's bound on those values
    rng = np.random.default_rng(6)
    K = 64
    Ac = rng.integers(0, 16, (3, K)).astype(np.uint8)
    Bc = rng.integers(0, 16, (4, K)).astype(np.uint8)
    As = np.full((3, 2), 127, np.uint8)
    Bs = np.full((4, 2), 127, np.uint8)
    A16 = gemm_ref.e2m1_decode(Ac).astype(np.float16)
    B16 = gemm_ref.e2m1_decode(Bc).astype(np.float16)
    C = rng.standard_normal((3, 4)).astype(np.float16)
    bias = rng.standard_normal(4).astype(np.float16)
    kw = dict(C=C, bias=bias, alpha=0.5, beta=-1.0, epilogue="bias_gelu")
    A, B = mx_ref.pack_e2m1(Ac), mx_ref.pack_e2m1(Bc)
    D = oracle.gemm_mx_reference(A, As, B, Bs, K, **kw)
    D16 = oracle.gemm_reference(A16, B16, K, **kw)
    assert np.array_equal(D, D16)
    assert np.array_equal(oracle.error_bound_mx(A, As, B, Bs, K, D, **kw),
                          oracle.error_bound(A16, B16, K, D16, **kw))
