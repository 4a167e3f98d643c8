"""Shared helpers of the GPU parity tests: move a workloads.Case to cuda:0,
run it through the C ABI, and compare with the oracle element by element."""

import numpy as np
import torch

import oracle


def to_device(case, dev="cuda:0", canary=0):
    """Device copies of the case's operands.  With canary > 0 the output buffer
    is allocated `canary` elements longer and the tail is returned separately
    so a test can check it is never written."""
    A = torch.from_numpy(np.ascontiguousarray(case.A)).to(dev)
    B = torch.from_numpy(np.ascontiguousarray(case.B)).to(dev)
    out_dtype = torch.int32 if case.dtype_a == "i8" else torch.float16
    n = case.M * case.N
    buf = torch.empty(n + canary, dtype=out_dtype, device=dev)
    if canary:
        fill = torch.full((canary,), 12345 if out_dtype == torch.int32 else -7.5, dtype=out_dtype)
        buf[n:] = fill.to(dev)
    C = buf[:n].view(case.M, case.N)
    if case.C is not None:
        C.copy_(torch.from_numpy(case.C).to(dev))
    else:
        C.zero_()
    bias = torch.from_numpy(case.bias).to(dev) if case.bias is not None else None
    return A, B, C, bias, buf


def run_case(dg, case, plan=None, stream=None, canary=0):
    A, B, C, bias, buf = to_device(case, canary=canary)
    dg.gemm(A, B, C, K=case.K, bias=bias, alpha=case.alpha, beta=case.beta,
            epilogue=case.epilogue, dtype_b=case.dtype_b, stream=stream, plan=plan)
    dg.check_status(stream)
    out = C.cpu().numpy()
    tail = buf[case.M * case.N:].cpu().numpy() if canary else None
    return out, tail


def run_case_ex(dg, case, ldc=None, ldd=None, inplace=False, stream=None):
    """Runs `case` through dg_gemm_ex with C and D in separate buffers of
    leading dimensions ldc and ldd (default N), or with D = C in place.  The
    columns between N and each leading dimension hold a canary; asserts that
    D's stay untouched and that C (with its padding) is unchanged."""
    dev = "cuda:0"
    M, N = case.M, case.N
    A = torch.from_numpy(np.ascontiguousarray(case.A)).to(dev)
    B = torch.from_numpy(np.ascontiguousarray(case.B)).to(dev)
    out_dtype = torch.int32 if case.dtype_a == "i8" else torch.float16
    fill = 12345 if out_dtype == torch.int32 else -7.5
    last = (case.program or [None])[-1]
    quant = isinstance(last, tuple) and last[0] == "quant_i8"
    ldd = ldd or N
    Dbuf = torch.full((M, ldd), 77 if quant else fill, dtype=torch.int8 if quant else out_dtype,
                      device=dev)
    D = Dbuf[:, :N]
    fill_d = 77 if quant else fill
    Cbuf = C = None
    if case.C is not None:
        if inplace:
            D.copy_(torch.from_numpy(case.C).to(dev))
            C = D
        else:
            Cbuf = torch.full((M, ldc or N), fill, dtype=out_dtype, device=dev)
            Cbuf[:, :N] = torch.from_numpy(case.C).to(dev)
            C = Cbuf[:, :N]
    c_before = Cbuf.cpu().numpy() if Cbuf is not None else None
    bias = torch.from_numpy(case.bias).to(dev) if case.bias is not None else None
    dg.gemm_ex(A, B, D, C=C, K=case.K, bias=bias, alpha=case.alpha, beta=case.beta,
               program=case.program or [], dtype_b=case.dtype_b, stream=stream)
    dg.check_status(stream)
    host = Dbuf.cpu().numpy()
    assert np.all(host[:, N:] == np.array(fill_d, dtype=host.dtype)), "D padding was written"
    if Cbuf is not None:
        assert np.array_equal(Cbuf.cpu().numpy().view(np.uint8), c_before.view(np.uint8)), \
            "C was modified"
    return host[:, :N]


def reference(case, rows=None):
    return oracle.gemm_reference(case.A, case.B, case.K, case.dtype_a, case.dtype_b, C=case.C,
                                 bias=case.bias, alpha=case.alpha, beta=case.beta,
                                 epilogue=case.epilogue, rows=rows, program=case.program)


def assert_parity(case, got, rows=None):
    """INT8: bit-exact.  Floating point: |D - D_ref| <= bound for every element."""
    ref = reference(case, rows)
    if rows is not None:
        got = got[rows]
    if case.dtype_a == "i8":
        bad = np.argwhere(got.astype(np.int64) != ref)
        assert bad.size == 0, "%s: %d mismatches, first at %s: got %d want %d" % (
            case.name, len(bad), tuple(bad[0]), got[tuple(bad[0])], ref[tuple(bad[0])])
        return
    bound = oracle.error_bound(case.A, case.B, case.K, ref, case.dtype_a, case.dtype_b, C=case.C,
                               bias=case.bias, alpha=case.alpha, beta=case.beta,
                               epilogue=case.epilogue, rows=rows, program=case.program)
    g = got.astype(np.float64)
    err = np.abs(g - ref)
    ok = err <= bound
    if not ok.all():
        idx = tuple(np.argwhere(~ok)[0])
        raise AssertionError(
            "%s: %d / %d elements outside the bound; first at %s: got %r want %r bound %r"
            % (case.name, int((~ok).sum()), ok.size, idx, g[idx], ref[idx], bound[idx]))
