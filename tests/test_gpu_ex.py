"""GPU parity of dg_gemm_ex: separate C and D with their own leading
dimensions, and epilogue programs, on every kernel family, against the CPU
oracle (floating point within oracle.error_bound, INT8 bit-exact).  Padding
columns of D hold a canary that must survive; C must come back unchanged."""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import assert_parity, run_case_ex

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    import __graft_entry__
    __graft_entry__.build()
    import precision_matmul_dg_gb300 as dg
    assert torch.cuda.is_available()
    return dg


PROGRAMS = {
    "empty": [],
    "bias_relu": ["bias", "relu"],
    "scale_gelu_clamp": [("scale", 0.5), "gelu", ("clamp", -0.1, 0.3)],
    "relu_bias_scale_clamp_gelu": ["relu", "bias", ("scale", -2.0), ("clamp", -1.0, 1.0), "gelu"],
    "eight_ops": ["bias", "gelu", ("scale", 1.5), "relu", ("clamp", 0.0, 2.0), ("scale", -1.0),
                  "gelu", "bias"],
}

# (dtypes, shape, kernel family the planner picks on a GB300)
FAMILIES = [
    (("f16", "f16"), (512, 1040, 520), "tc, single CTA"),
    (("f16", "f16"), (1536, 2000, 512), "tc, CTA pair"),
    (("f16", "f16"), (128, 4096, 16384), "tc, stream-K (two K halves per tile)"),
    (("f16", "f16"), (3, 300, 5000), "gemv, split-K"),
    (("f16", "f16"), (1, 4000, 3000), "gemv"),
    (("f16", "f16"), (5, 1000, 3000), "warp-MMA gemv"),
    (("f16", "f16"), (16, 700, 20000), "warp-MMA gemv, split-K"),
    (("f16", "e2m1"), (8, 1000, 2048), "skinny"),
    (("f16", "e2m1"), (130, 1000, 512), "tc with in-kernel widening"),
    (("f16", "e2m1"), (1024, 2048, 1024), "tc, weights widened in tensor memory"),
    (("f16", "e2m1"), (2048, 2048, 1024), "widened then tc pair"),
]


def _case(dtypes, shape, program, beta, seed):
    M, N, K = shape
    return workloads.random_case(M, N, K, dtype_a=dtypes[0], dtype_b=dtypes[1], alpha=-0.75,
                                 beta=beta, seed=seed, program=program, pad=float("nan"))


def _rows(case):
    # the oracle on every row for small outputs, on a spread of rows otherwise
    if case.M * case.N * case.K <= 2e9:
        return None
    return np.unique(np.concatenate([np.arange(0, case.M, 97), [case.M - 1]]))


@pytest.mark.parametrize("fam", FAMILIES, ids=lambda f: f[2])
@pytest.mark.parametrize("prog", sorted(PROGRAMS))
def test_programs_every_family(dg, fam, prog):
    dtypes, shape, _ = fam
    case = _case(dtypes, shape, PROGRAMS[prog], 0.5, hash((shape, prog)) % 1000)
    N = case.N
    got = run_case_ex(dg, case, ldc=N + 8, ldd=N + 24)
    assert_parity(case, got, _rows(case))


@pytest.mark.parametrize("fam", FAMILIES, ids=lambda f: f[2])
@pytest.mark.parametrize("layout", ["in_place", "no_c", "odd_ldd", "odd_ldc", "wide_both"])
def test_layouts_every_family(dg, fam, layout):
    dtypes, shape, _ = fam
    prog = PROGRAMS["relu_bias_scale_clamp_gelu"]
    beta = 0.0 if layout == "no_c" else -1.25
    case = _case(dtypes, shape, prog, beta, 17)
    N = case.N
    kw = {"in_place": dict(inplace=True, ldd=N + 16),
          "no_c": dict(ldd=N + 8),
          "odd_ldd": dict(ldc=N, ldd=N + 3),     # D rows not 16-byte aligned: direct stores
          "odd_ldc": dict(ldc=N + 1, ldd=N),     # C rows not 16-byte aligned: direct loads
          "wide_both": dict(ldc=2 * N + 8, ldd=3 * N + 40)}[layout]
    got = run_case_ex(dg, case, **kw)
    assert_parity(case, got, _rows(case))


@pytest.mark.parametrize("shape", [(256, 520, 640), (64, 300, 200), (3, 1000, 1000),
                                   (4096, 4096, 4096)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout", ["separate", "in_place", "odd_ld"])
def test_int8_separate_d(dg, shape, layout):
    M, N, K = shape
    case = workloads.random_case(M, N, K, dtype_a="i8", dtype_b="i8", alpha=3.0, beta=-2.0,
                                 seed=23)
    kw = {"separate": dict(ldc=N + 4, ldd=N + 12), "in_place": dict(inplace=True, ldd=N + 4),
          "odd_ld": dict(ldc=N + 1, ldd=N + 3)}[layout]
    got = run_case_ex(dg, case, **kw)
    assert_parity(case, got, _rows(case))


def test_k_zero_program(dg):
    for dtypes in (("f16", "f16"), ("i8", "i8")):
        prog = ["bias", ("scale", 2.0), "relu"] if dtypes[0] == "f16" else []
        case = workloads.random_case(33, 70, 8, dtype_a=dtypes[0], dtype_b=dtypes[1], beta=0.5
                                     if dtypes[0] == "f16" else 3.0, seed=3, program=prog)
        case.K = 0
        got = run_case_ex(dg, case, ldc=72, ldd=75)
        assert_parity(case, got)


def test_program_extremes(dg):
    # results on both sides of every clamp bound, exact zeros from ReLU, and a
    # scale that takes values near the FP16 maximum
    case = _case(("f16", "f16"), (300, 520, 200), [("scale", 3000.0), ("clamp", -60000.0, 2000.0),
                                                   "relu"], 0.5, 41)
    got = run_case_ex(dg, case, ldc=520, ldd=528)
    assert_parity(case, got)
    assert (got == 0).mean() > 0.3 and (got == np.float16(2000.0)).mean() > 0.05


QUANT_PROGRAMS = {
    "quant": [("quant_i8", 40.0)],
    "bias_gelu_quant": ["bias", "gelu", ("quant_i8", 60.0)],
    "relu_clamp_quant": ["relu", ("clamp", 0.0, 1.5), ("quant_i8", 84.6)],
    "saturating": [("scale", 7.0), ("quant_i8", 100.0)],
}


@pytest.mark.parametrize("fam", FAMILIES, ids=lambda f: f[2])
@pytest.mark.parametrize("prog", sorted(QUANT_PROGRAMS))
def test_int8_output_every_family(dg, fam, prog):
    # int8 D (program ending in a quantization): codes within |a| E + 1 of
    # the oracle's, where E bounds the error of t; D padding untouched
    dtypes, shape, _ = fam
    case = _case(dtypes, shape, QUANT_PROGRAMS[prog], 0.5, hash((shape, prog)) % 997)
    N = case.N
    layout = dict(ldc=N + 8, ldd=N + 16) if "bias" in prog else dict(ldc=N, ldd=N + 5)
    got = run_case_ex(dg, case, **layout)
    assert got.dtype == np.int8
    assert_parity(case, got.astype(np.float64), _rows(case))
    if prog == "saturating":
        assert (got == 127).any() and (got == -128).any()


def test_int8_output_rejects_in_place(dg):
    case = _case(("f16", "f16"), (64, 128, 64), [("quant_i8", 1.0)], 0.5, 3)
    A = torch.from_numpy(case.A).cuda()
    B = torch.from_numpy(case.B).cuda()
    C = torch.from_numpy(case.C).cuda()
    with pytest.raises(dg.DgError):
        dg.gemm_ex_raw(64, 128, 64, "f16", "f16", A, case.lda, B, case.ldb, C, 128, C, 128, None,
                       1.0, 0.5, program=[("quant_i8", 1.0)])


def test_fixed_epilogue_equals_program(dg):
    # dg_gemm's bias+GELU form and the program ["bias", "gelu"] are the same
    # function: both must meet the oracle on the same inputs
    for shape in [(512, 1040, 520), (3, 300, 5000), (8, 1000, 2048)]:
        dtypes = ("f16", "e2m1") if shape[0] == 8 else ("f16", "f16")
        case = _case(dtypes, shape, ["bias", "gelu"], 0.5, 5)
        got = run_case_ex(dg, case, ldc=shape[1], ldd=shape[1])
        assert_parity(case, got)
        fixed = workloads.random_case(*shape, dtype_a=dtypes[0], dtype_b=dtypes[1], alpha=-0.75,
                                      beta=0.5, seed=5, epilogue="bias_gelu", pad=float("nan"))
        np.testing.assert_array_equal(fixed.bias, case.bias)
        from gpu_util import run_case
        got2, _ = run_case(dg, fixed)
        assert_parity(fixed, got2)
