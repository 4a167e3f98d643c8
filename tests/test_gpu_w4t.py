"""W4A16 with the packed weights widened in tensor memory, against the oracle.

The kernel computes D^T tiles of 128 weight rows x 160 activation rows: the
weights are the MMA's A operand, widened code by code into tensor memory,
and each epilogue lane writes one column of D.  The bound is the FP16
path's (oracle.error_bound): every E2M1 value is exact in FP16.
"""

import os

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


def _w4t_plans(dg, case):
    plans = [p for p in dg.plan_tiles(case.M, case.N, case.K, "f16", "e2m1", case.epilogue,
                                      target_occupancy=0.0)
             if p["kernel_name"] == "tc" and p["swap_ab"]]
    assert sorted(p["n_tile"] for p in plans) == [160, 224]
    return plans


def _w4t_plan(dg, case, n_tile=160):
    return [p for p in _w4t_plans(dg, case) if p["n_tile"] == n_tile][0]


# ragged M, N and K (odd K: a half byte past the last code of each row), M
# below one activation tile, N below one weight tile, several tiles per CTA
SHAPES = [(200, 700, 600), (161, 129, 64), (1000, 264, 1536), (7, 300, 99), (640, 1000, 130),
          (2048, 2176, 512)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("epi", ["none", "bias", "gelu", "bias_gelu"])
def test_w4t_shapes(dg, shape, epi):
    M, N, K = shape
    case = workloads.random_case(M, N, K, "f16", "e2m1", epilogue=epi, alpha=0.75, beta=-0.5,
                                 seed=hash((M, N, K, epi)) % 991, pad=255)
    for p in _w4t_plans(dg, case):
        for grid in (p["grid"], 5, 1):  # persistent CTAs walking several tiles
            got, _ = run_case(dg, case, plan=dict(p, grid=grid))
            assert_parity(case, got)


def test_w4t_without_c(dg):
    case = workloads.random_case(900, 1100, 768, "f16", "e2m1", epilogue="bias_gelu", seed=21)
    for p in _w4t_plans(dg, case):
        got, tail = run_case(dg, case, plan=p, canary=64)
        assert_parity(case, got)
        assert np.all(tail == np.float16(-7.5))


def test_w4t_every_code_one_hot(dg):
    """Column j of the weights holds code j % 16 at k = j % K and zeros
    elsewhere, so D[:, j] = A[:, k] * value(code): each decoded value appears
    exactly (table from the pinned golden file)."""
    table = {}
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "e2m1_codes.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            c, v = line.split()
            table[int(c)] = float(v)
    M, N, K = 200, 192, 128
    case = workloads.random_case(M, N, K, "f16", "e2m1", seed=4)
    case.A = np.ascontiguousarray(np.round(case.A * 8) / 8).astype(np.float16)
    packed = np.zeros_like(case.B)
    for j in range(N):
        k, code = j % K, j % 16
        packed[j, k // 2] |= np.uint8(code << (4 * (k % 2)))
    case.B = packed
    for p in _w4t_plans(dg, case):
        got, _ = run_case(dg, case, plan=p)
        for j in range(N):
            want = case.A[:, j % K].astype(np.float64) * table[j % 16]
            assert np.array_equal(got[:, j].astype(np.float64), want), j


@pytest.mark.parametrize("n_tile", [160, 224])
def test_w4t_full_size(dg, n_tile):
    case = workloads.WORKLOADS["w4a16_m2048"]()
    a, _ = run_case(dg, case, plan=_w4t_plan(dg, case, n_tile))
    assert_parity(case, a)
    b, _ = run_case(dg, case, plan=_w4t_plan(dg, case, n_tile))
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))  # fixed summation order


def test_w4t_unaligned_output_takes_the_widening_path(dg):
    # rows of D that are not 16-byte multiples (N = 501): the plan runs the
    # widening pre-pass and the FP16 kernel instead
    case = workloads.random_case(300, 501, 600, "f16", "e2m1", epilogue="bias", beta=0.5,
                                 seed=6, pad=255)
    got, _ = run_case(dg, case, plan=_w4t_plan(dg, case))
    assert_parity(case, got)
