"""GPU parity of dg_gemm_strided_batched against the CPU oracle, problem by
problem (floating point within oracle.error_bound, INT8 bit-exact)."""

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


def _problems(batch, M, N, K, dtype_a="f16", dtype_b="f16", epilogue="none", alpha=1.0,
              beta=0.0, shared_b=False, shared_bias=False, seed=0):
    """`batch` seeded cases of one shape (as workloads.random_case)."""
    cases = [workloads.random_case(M, N, K, dtype_a, dtype_b, epilogue=epilogue, alpha=alpha,
                                   beta=beta, seed=seed * 1000 + z) for z in range(batch)]
    if shared_b:
        for c in cases:
            c.B = cases[0].B
    if shared_bias and cases[0].bias is not None:
        for c in cases:
            c.bias = cases[0].bias
    return cases


def _run(dg, cases, shared_b=False, shared_bias=False, stream=None):
    dev = "cuda:0"
    c0 = cases[0]
    A = torch.from_numpy(np.stack([c.A for c in cases])).to(dev)
    B = torch.from_numpy(c0.B if shared_b else np.stack([c.B for c in cases])).to(dev)
    out = torch.int32 if c0.dtype_a == "i8" else torch.float16
    C = torch.zeros(len(cases), c0.M, c0.N, dtype=out, device=dev)
    if c0.C is not None:
        C.copy_(torch.from_numpy(np.stack([c.C for c in cases])))
    bias = None
    if c0.bias is not None:
        bias = torch.from_numpy(c0.bias if shared_bias else np.stack([c.bias for c in cases]))
        bias = bias.to(dev)
    dg.gemm_batched(A, B, C, K=c0.K, bias=bias, alpha=c0.alpha, beta=c0.beta,
                    epilogue=c0.epilogue, dtype_b=c0.dtype_b, stream=stream)
    dg.check_status(stream)
    return C.cpu().numpy()


def _check(cases, got):
    for z, c in enumerate(cases):
        ref = oracle.gemm_reference(c.A, c.B, c.K, c.dtype_a, c.dtype_b, C=c.C, bias=c.bias,
                                    alpha=c.alpha, beta=c.beta, epilogue=c.epilogue)
        if c.dtype_a == "i8":
            assert np.array_equal(got[z].astype(np.int64), ref), "problem %d" % z
            continue
        bound = oracle.error_bound(c.A, c.B, c.K, ref, c.dtype_a, c.dtype_b, C=c.C, bias=c.bias,
                                   alpha=c.alpha, beta=c.beta, epilogue=c.epilogue)
        err = np.abs(got[z].astype(np.float64) - ref)
        assert (err <= bound).all(), "problem %d: %d elements outside the bound" % (
            z, int((err > bound).sum()))


def test_qkv_projections_one_launch(dg):
    # 96 problems of 1 x 128 x 4096: the GEMV takes them in one launch
    cases = _problems(96, 1, 128, 4096, epilogue="bias", seed=1)
    before = dg.launch_count()
    got = _run(dg, cases)
    assert dg.launch_count() - before == 1
    _check(cases, got)


@pytest.mark.parametrize("shape", [(3, 300, 20000), (8, 200, 777), (1, 4096, 65536),
                                   (5, 100, 8)], ids=lambda s: "x".join(map(str, s)))
def test_gemv_batches(dg, shape):
    # split-K GEMV problems; shared B and shared bias
    M, N, K = shape
    cases = _problems(7, M, N, K, epilogue="bias_gelu", alpha=-0.5, beta=1.5, shared_b=True,
                      shared_bias=True, seed=2)
    got = _run(dg, cases, shared_b=True, shared_bias=True)
    _check(cases, got)


def test_batch_above_grid_limit(dg):
    # more problems than one launch's grid.z takes (65535)
    batch, M, N, K = 66000, 1, 8, 16
    g = np.random.default_rng(3)
    A = g.standard_normal((batch, M, K)).astype(np.float16)
    B = g.standard_normal((batch, N, K)).astype(np.float16)
    dev = "cuda:0"
    C = torch.zeros(batch, M, N, dtype=torch.float16, device=dev)
    dg.gemm_batched(torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev), C)
    dg.check_status()
    got = C.cpu().numpy().astype(np.float64)
    for z in list(range(0, batch, 997)) + [65534, 65535, 65536, batch - 1]:
        ref = oracle.gemm_reference(A[z], B[z], K)
        bound = oracle.error_bound(A[z], B[z], K, ref)
        assert (np.abs(got[z] - ref) <= bound).all(), z


@pytest.mark.parametrize("kind", ["tc_f16", "tc_f16_ragged", "w4a16_skinny", "w4a16_tc", "int8",
                                  "int8_ragged", "k_zero"])
def test_batches_on_other_kernels(dg, kind):
    # shapes the planner sends to other kernels: one launch per problem.  The
    # ragged shapes pack outputs of M*N elements with M*N odd, so problem 1's
    # C and D start off any 16-byte boundary.
    if kind == "tc_f16":
        cases = _problems(3, 256, 520, 200, epilogue="bias_gelu", beta=0.5, seed=4)
    elif kind == "tc_f16_ragged":
        cases = _problems(3, 255, 521, 200, epilogue="bias_gelu", beta=0.5, seed=10)
    elif kind == "int8_ragged":
        cases = _problems(3, 255, 521, 640, "i8", "i8", alpha=-1.0, beta=5.0, seed=11)
    elif kind == "w4a16_skinny":
        cases = _problems(4, 8, 1000, 2048, "f16", "e2m1", epilogue="bias", seed=5)
    elif kind == "w4a16_tc":
        cases = _problems(3, 300, 600, 200, "f16", "e2m1", epilogue="gelu", beta=-1.0, seed=6)
    elif kind == "int8":
        cases = _problems(3, 256, 520, 640, "i8", "i8", alpha=3.0, beta=-2.0, seed=7)
    else:
        cases = _problems(3, 33, 70, 8, epilogue="bias", beta=0.5, seed=8)
        for c in cases:
            c.K = 0
    got = _run(dg, cases)
    _check(cases, got)


def test_batch_of_one_equals_gemm(dg):
    case = workloads.random_case(3, 300, 5000, epilogue="gelu", beta=0.5, seed=9)
    got = _run(dg, [case])
    from gpu_util import run_case
    ref, _ = run_case(dg, case)
    assert np.array_equal(got[0].view(np.uint16), ref.view(np.uint16))
