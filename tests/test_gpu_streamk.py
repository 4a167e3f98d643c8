"""Stream-K work division of the FP16 tensor-core kernel against the oracle.

The tiles that leave the last wave ragged have their K blocks dealt out in
even ranges, one per CTA (pair); a tile split between ranges is finished by
the range holding its first K block, which adds the other ranges' FP32
partials in piece order.  The bound is the FP16 path's (oracle.error_bound):
splitting K only changes the order of FP32 additions.
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


def _sk_plans(dg, M, N, K):
    return [p for p in dg.plan_tiles(M, N, K, target_occupancy=0.0)
            if p["kernel_name"] == "tc_streamk"]


# (M, N, K): tiles cut into two to four pieces, ragged M, N and K, a short
# K (ranges near the 4-block minimum); N % 8 == 0 (16-byte rows of D, as the
# staged epilogue needs).  With 7 and 3 units the tiles outnumber the units:
# whole tiles, then ranges that straddle tiles
SHAPES = [(520, 1096, 700), (300, 520, 520), (129, 264, 4096), (1000, 24, 999),
          (640, 768, 4096), (512, 1024, 512)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("epi", ["none", "bias_gelu"])
def test_stream_k_parity(dg, shape, epi):
    M, N, K = shape
    case = workloads.random_case(M, N, K, epilogue=epi, alpha=1.5, beta=0.25,
                                 seed=hash((M, N, K, epi)) % 997, pad=float("nan"))
    plans = _sk_plans(dg, M, N, K)
    assert plans, "a ragged shape has stream-K plans"
    for p in plans:
        # the planner's grid, and fewer units: whole tiles then ranges
        for units in (p["grid"] // p["cta_group"], 7, 3):
            q = dict(p, grid=units * p["cta_group"])
            got, _ = run_case(dg, case, plan=q)
            assert_parity(case, got)


def test_stream_k_without_c(dg):
    # beta = 0: the finishing range stores only; canary past D untouched
    case = workloads.random_case(700, 904, 520, epilogue="bias_gelu", alpha=-1.25, seed=12)
    for p in _sk_plans(dg, 700, 904, 520):
        got, tail = run_case(dg, case, plan=p, canary=64)
        assert_parity(case, got)
        assert np.all(tail == np.float16(-7.5))


def test_stream_k_bit_stable(dg):
    # the partials are added in a fixed order: repeated launches agree bit
    # for bit, whichever range finishes first
    case = workloads.random_case(1000, 1000, 3000, beta=0.5, seed=2)
    for p in _sk_plans(dg, 1000, 1000, 3000):
        outs = [run_case(dg, case, plan=p)[0] for _ in range(3)]
        assert_parity(case, outs[0])
        for o in outs[1:]:
            assert np.array_equal(o.view(np.uint16), outs[0].view(np.uint16))


def test_stream_k_back_to_back(dg):
    # launches on one stream with no host synchronisation between them, each
    # on new data and some on another shape (the workspace grows): a flag or
    # a partial of an earlier launch is never taken for this launch's
    dev = "cuda:0"
    shapes = [(520, 1096, 700), (520, 1096, 700), (512, 1024, 512), (300, 520, 520),
              (520, 1096, 700)]
    cases = [workloads.random_case(*s, beta=0.5, epilogue="bias", seed=40 + i)
             for i, s in enumerate(shapes)]
    outs = []
    for case in cases:
        p = [q for q in _sk_plans(dg, case.M, case.N, case.K) if q["cta_group"] == 2][0]
        A = torch.from_numpy(case.A).to(dev)
        B = torch.from_numpy(case.B).to(dev)
        C = torch.from_numpy(case.C).to(dev)
        bias = torch.from_numpy(case.bias).to(dev)
        dg.gemm(A, B, C, K=case.K, bias=bias, alpha=case.alpha, beta=case.beta,
                epilogue=case.epilogue, plan=p)
        outs.append(C)
    dg.check_status()
    for case, C in zip(cases, outs):
        assert_parity(case, C.cpu().numpy())


def test_stream_k_unaligned_output_runs_whole_tiles(dg):
    # rows of D that are not 16-byte aligned (N = 1100) leave the staged
    # epilogue out: the stream-K plan runs the data-parallel kernel of its tile
    case = workloads.random_case(520, 1100, 700, epilogue="bias_gelu", beta=0.5, seed=3)
    for p in _sk_plans(dg, 520, 1100, 700):
        got, _ = run_case(dg, case, plan=p)
        assert_parity(case, got)


def test_stream_k_single_k_block(dg):
    # one K block per tile: nothing to split, whole tiles
    case = workloads.random_case(900, 704, 40, epilogue="gelu", beta=-0.5, seed=8)
    for p in _sk_plans(dg, 900, 704, 4096):
        got, _ = run_case(dg, case, plan=p)
        assert_parity(case, got)
