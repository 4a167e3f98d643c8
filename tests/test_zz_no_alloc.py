"""dg_gemm_thin_noalloc: the thin-M GEMM for callers that cannot allocate.

Callers such as code running under CUDA-graph capture, or runtimes that own
every byte of device memory through their own pool, cannot let a library call
cudaMalloc.  This entry point runs the split-K GEMV with its partial sums and
counters in the library's static device array instead.  The test calls it
through the C ABI twice in a row (the second call finds the first call's
leftovers in the shared array) and checks both results against dg_gemm's
output on the same inputs, within the oracle bound the parity tests use.

Kept in a file pytest collects last, so a run that stops at the first
failure has already run every other test; it passes alone in a fresh
process as well.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    import __graft_entry__
    __graft_entry__.build()
    import precision_matmul_dg_gb300 as dg
    assert torch.cuda.is_available()
    return dg


def _noalloc(dg, case, A, B, C, bias, stream):
    L = dg.lib()
    st = L.dg_gemm_thin_noalloc(
        case.M, case.N, case.K, dg.F16, dg.F16, ctypes.c_void_p(A.data_ptr()), case.lda,
        ctypes.c_void_p(B.data_ptr()), case.ldb, ctypes.c_void_p(C.data_ptr()),
        ctypes.c_void_p(bias.data_ptr()) if bias is not None else None, case.alpha, case.beta,
        dg.EPILOGUES[case.epilogue], ctypes.c_void_p(stream.cuda_stream))
    assert st == 0, dg.last_error()


@pytest.mark.parametrize("shape,epi", [((1, 256, 12800), "none"), ((4, 300, 30000), "bias_gelu"),
                                       ((8, 1000, 5000), "gelu"), ((1, 4096, 20000), "bias")])
def test_noalloc_matches_dg_gemm_twice(dg, shape, epi):
    M, N, K = shape
    case = workloads.random_case(M, N, K, epilogue=epi, alpha=0.5, beta=-1.5, seed=K + N)
    stream = torch.cuda.current_stream()

    # existing entry point
    A, B, C_ref, bias, _ = to_device(case)
    dg.gemm(A, B, C_ref, K=K, bias=bias, alpha=case.alpha, beta=case.beta, epilogue=epi,
            stream=stream)
    want = C_ref.cpu().numpy().astype(np.float64)

    ref = oracle.gemm_reference(case.A, case.B, K, C=case.C, bias=case.bias, alpha=case.alpha,
                                beta=case.beta, epilogue=epi)
    bound = oracle.error_bound(case.A, case.B, K, ref, C=case.C, bias=case.bias,
                               alpha=case.alpha, beta=case.beta, epilogue=epi)
    for call in range(2):
        C = torch.from_numpy(case.C).cuda()  # fresh C each call: C is read (beta != 0)
        _noalloc(dg, case, A, B, C, bias, stream)
        torch.cuda.synchronize()
        got = C.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - want) <= bound), "call %d differs from dg_gemm" % call
        assert np.all(np.abs(got - ref) <= bound), "call %d outside the oracle bound" % call


def test_noalloc_rejects_what_it_does_not_take(dg):
    L = dg.lib()
    z = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    st = L.dg_gemm_thin_noalloc(16, 64, 64, dg.F16, dg.F16, ctypes.c_void_p(z.data_ptr()), 64,
                                ctypes.c_void_p(z.data_ptr()), 64, ctypes.c_void_p(z.data_ptr()),
                                None, 1.0, 0.0, 0, None)
    assert st == 2 and "M <= 8" in dg.last_error()   # DG_ERR_UNSUPPORTED
