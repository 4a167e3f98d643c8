"""The widening path on CTA pairs, against the oracle.

Plans of 256 x 192 CTA-pair tiles on the widening path (INT8 operands with
exact INT32 output, E2M1 weights with FP16 output), and the INT8 plan of
256 x 224 tiles (whose last 32-column chunk keeps its running INT32 sums in
a staging box during the tile, 16 columns per epilogue warp): the narrow
operands are
widened into FP16 copies and the pair kernel reads them.  These tests run
that plan on ragged shapes, on K below, at and across 512, on padded source
rows and on grids from one CTA pair (which walks every tile) to the
planner's, and queue launches of other sizes and types in between; INT8
results are bit-exact, FP16 within the FP16 path's bound.
"""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import assert_parity, run_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    import __graft_entry__
    __graft_entry__.build()
    import precision_matmul_dg_gb300 as dg
    assert torch.cuda.is_available()
    return dg


def _pair192(dg, case, n_tile=192):
    plans = [p for p in dg.plan_tiles(case.M, case.N, case.K, case.dtype_a, case.dtype_b,
                                      case.epilogue, target_occupancy=0.0)
             if p["kernel_name"] == "tc_widened" and p["n_tile"] == n_tile and p["cta_group"] == 2]
    assert len(plans) == 1, plans
    return plans[0]


# a last row panel of one row (the second CTA of that pair has none), K below
# 512, K = 1 and odd K, K across 512 with a ragged rest, N ragged
SHAPES = [(300, 501, 600), (1000, 700, 99), (257, 193, 1), (130, 1000, 2500), (600, 390, 1030),
          (2048, 2048, 1536), (129, 385, 513)]
GRIDS = (None, 2, 6, 22)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("n_tile", [192, 224])
def test_int8_widened_pair(dg, shape, n_tile):
    M, N, K = shape
    case = workloads.random_case(M, N, K, "i8", "i8", alpha=3, beta=-2,
                                 seed=hash(shape) % 997, pad=127)
    p = _pair192(dg, case, n_tile)
    for grid in GRIDS:
        got, _ = run_case(dg, case, plan=p if grid is None else dict(p, grid=grid))
        assert_parity(case, got)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("epi", ["none", "bias_gelu"])
def test_w4a16_widened_pair(dg, shape, epi):
    M, N, K = shape
    case = workloads.random_case(M, N, K, "f16", "e2m1", epilogue=epi, alpha=0.75, beta=0.5,
                                 seed=hash((shape, epi)) % 991, pad=255)
    p = _pair192(dg, case)
    for grid in GRIDS:
        got, _ = run_case(dg, case, plan=p if grid is None else dict(p, grid=grid))
        assert_parity(case, got)


def test_padded_sources(dg):
    # source rows longer than K (the padding holds values the copy must not
    # carry into the product)
    case = workloads.random_case(700, 900, 1000, "i8", "i8", lda=1056, ldb=1024, seed=8,
                                 pad=-128)
    got, _ = run_case(dg, case, plan=_pair192(dg, case))
    assert_parity(case, got)
    case = workloads.random_case(700, 900, 1001, "f16", "e2m1", ldb=1088, seed=9, pad=255)
    got, _ = run_case(dg, case, plan=_pair192(dg, case))
    assert_parity(case, got)


def test_alternating_shapes_and_types(dg):
    # launches of other sizes and the other operand type in between reuse the
    # same widening workspace
    cases = [workloads.random_case(1500, 1200, 2100, "i8", "i8", seed=11),
             workloads.random_case(300, 400, 300, "f16", "e2m1", seed=12),
             workloads.random_case(2100, 1700, 700, "f16", "e2m1", epilogue="bias", seed=13),
             workloads.random_case(200, 260, 5000, "i8", "i8", beta=1, seed=14)]
    plans = [_pair192(dg, c) for c in cases]
    for _ in range(2):
        for c, p in zip(cases, plans):
            got, _ = run_case(dg, c, plan=p)
            assert_parity(c, got)


@pytest.mark.parametrize("n_tile", [192, 224])
def test_int8_widened_pair_extremes(dg, n_tile):
    # every product -128 * -128 through the widened copies: chunk sums of
    # exactly 2^24, and the INT32 result exact (D rows 16-byte multiples: the
    # staged stores; rows of 454 are not, and take the direct stores)
    K = 4096
    for N in (576, 454):
        case = workloads.random_case(512, N, K, "i8", "i8", seed=1)
        case.A = np.full_like(case.A, -128)
        case.B = np.full_like(case.B, -128)
        got, _ = run_case(dg, case, plan=_pair192(dg, case, n_tile))
        assert np.all(got == 128 * 128 * K)


@pytest.mark.parametrize("n_tile", [192, 224])
def test_int8_column_one_hot(dg, n_tile):
    # D[:, j] = A[:, j % K] * B[j, j % K]: every column of a tile, including
    # the split chunk's 32 (columns 192 .. 223 of each 224-wide tile), lands
    # where it belongs
    M, N, K = 300, 700, 1100
    case = workloads.random_case(M, N, K, "i8", "i8", seed=17)
    B = np.zeros_like(case.B)
    for j in range(N):
        B[j, j % K] = (j % 255) - 127
    case.B = B
    got, _ = run_case(dg, case, plan=_pair192(dg, case, n_tile))
    want = case.A[:, np.arange(N) % K].astype(np.int64) * B[np.arange(N), np.arange(N) % K]
    assert np.array_equal(got.astype(np.int64), want)


def test_back_to_back_in_one_stream(dg):
    # many launches queued without a host sync in between, each rewriting the
    # copies the one before read (programmatic dependent launches)
    case = workloads.random_case(1024, 1344, 1536, "f16", "e2m1", epilogue="bias_gelu", seed=15)
    p = _pair192(dg, case)
    A = torch.from_numpy(case.A).cuda()
    B = torch.from_numpy(case.B).cuda()
    bias = torch.from_numpy(case.bias).cuda()
    outs = [torch.empty(case.M, case.N, dtype=torch.float16, device="cuda") for _ in range(6)]
    for D in outs:
        dg.gemm(A, B, D, K=case.K, bias=bias, epilogue=case.epilogue, dtype_b="e2m1", plan=p)
    dg.check_status()
    first = outs[0].cpu().numpy()
    assert_parity(case, first)
    for D in outs[1:]:
        assert np.array_equal(D.cpu().numpy().view(np.uint16), first.view(np.uint16))
