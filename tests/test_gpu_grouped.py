"""GPU parity of dg_gemm_grouped (problems of one N and K with their own M and
buffers) against the CPU oracle, problem by problem."""

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    import __graft_entry__
    __graft_entry__.build()
    import precision_matmul_dg_gb300 as dg
    assert torch.cuda.is_available()
    return dg


def _group(Ms, N, K, dtype_a="f16", dtype_b="f16", epilogue="none", alpha=1.0, beta=0.0,
           shared_b=False, seed=0):
    cases = [workloads.random_case(max(m, 1), N, K, dtype_a, dtype_b, epilogue=epilogue,
                                   alpha=alpha, beta=beta, seed=seed * 100 + g)
             for g, m in enumerate(Ms)]
    for c, m in zip(cases, Ms):
        c.M = m
        c.A = c.A[:m]
        if c.C is not None:
            c.C = c.C[:m]
    if shared_b:
        for c in cases:
            c.B = cases[0].B
    if cases[0].bias is not None:
        for c in cases:
            c.bias = cases[0].bias
    return cases


def _run(dg, cases, shared_b=False):
    dev = "cuda:0"
    out = torch.int32 if cases[0].dtype_a == "i8" else torch.float16
    As = [torch.from_numpy(np.ascontiguousarray(c.A)).to(dev) for c in cases]
    Bs = (torch.from_numpy(cases[0].B).to(dev) if shared_b else
          [torch.from_numpy(c.B).to(dev) for c in cases])
    Cs = []
    for c in cases:
        C = torch.zeros(c.M, c.N, dtype=out, device=dev)
        if c.C is not None and c.M:
            C.copy_(torch.from_numpy(c.C))
        Cs.append(C)
    bias = torch.from_numpy(cases[0].bias).to(dev) if cases[0].bias is not None else None
    c0 = cases[0]
    dg.gemm_grouped(As, Bs, Cs, K=c0.K, bias=bias, alpha=c0.alpha, beta=c0.beta,
                    epilogue=c0.epilogue)
    dg.check_status()
    return [C.cpu().numpy() for C in Cs]


def _check(cases, got):
    for g, c in enumerate(cases):
        if c.M == 0:
            assert got[g].size == 0
            continue
        ref = oracle.gemm_reference(c.A, c.B, c.K, c.dtype_a, c.dtype_b, C=c.C, bias=c.bias,
                                    alpha=c.alpha, beta=c.beta, epilogue=c.epilogue)
        if c.dtype_a == "i8":
            assert np.array_equal(got[g].astype(np.int64), ref), g
            continue
        bound = oracle.error_bound(c.A, c.B, c.K, ref, c.dtype_a, c.dtype_b, C=c.C, bias=c.bias,
                                   alpha=c.alpha, beta=c.beta, epilogue=c.epilogue)
        assert (np.abs(got[g].astype(np.float64) - ref) <= bound).all(), "problem %d" % g


def test_experts_one_launch(dg):
    # eight experts with 0..16 routed rows: one launch of the warp-MMA GEMV
    cases = _group([0, 1, 3, 7, 16, 5, 12, 2], 512, 2048, epilogue="bias_gelu", beta=0.5,
                   seed=1)
    before = dg.launch_count()
    got = _run(dg, cases)
    assert dg.launch_count() - before == 1
    _check(cases, got)


@pytest.mark.parametrize("K", [8, 100, 4097, 20000])
def test_split_k_groups(dg, K):
    cases = _group([3, 16, 1, 9], 300, K, epilogue="gelu", alpha=-0.5, beta=1.25,
                   shared_b=True, seed=2)
    got = _run(dg, cases, shared_b=True)
    _check(cases, got)


@pytest.mark.parametrize("kind", ["large_m", "e2m1", "int8"])
def test_groups_on_other_kernels(dg, kind):
    # a problem with M > 16, or another dtype pair: one launch per problem
    if kind == "large_m":
        cases = _group([4, 200, 0, 17], 256, 512, epilogue="bias", beta=0.5, seed=3)
    elif kind == "e2m1":
        cases = _group([8, 300], 512, 1024, "f16", "e2m1", epilogue="bias_gelu", seed=4)
    else:
        cases = _group([5, 130], 256, 640, "i8", "i8", alpha=2.0, beta=-1.0, seed=5)
    got = _run(dg, cases)
    _check(cases, got)


def test_prepared_group_runs_again_on_new_data(dg):
    # prepare_grouped builds the pointer arrays once; running it again after
    # the inputs changed in place gives the new product (the bench's
    # mixture-of-experts workload runs this way)
    from gpu_util import assert_parity
    Ms = [3, 0, 16, 7, 1]
    first = _group(Ms, 520, 1000, seed=8)
    second = _group(Ms, 520, 1000, seed=9)
    dev = "cuda:0"
    As = [torch.from_numpy(np.ascontiguousarray(c.A)).to(dev) for c in first]
    Bs = [torch.from_numpy(c.B).to(dev) for c in first]
    Cs = [torch.zeros(c.M, c.N, dtype=torch.float16, device=dev) for c in first]
    run = dg.prepare_grouped(As, Bs, Cs, K=1000)
    for cases in (first, second):
        for c, A, B in zip(cases, As, Bs):
            A.copy_(torch.from_numpy(np.ascontiguousarray(c.A)))
            B.copy_(torch.from_numpy(c.B))
        run()
        dg.check_status()
        for c, C in zip(cases, Cs):
            if c.M:
                assert_parity(c, C.cpu().numpy())
