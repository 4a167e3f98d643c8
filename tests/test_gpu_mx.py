"""GPU parity of the MXFP4 entry points against the CPU oracle:
dg_quantize_mxf4 bit-exact (codes and scale bytes, bytes past the row's end
untouched), and dg_gemm_mxf4 within the oracle's floating-point bound."""

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

CANARY = 0xAB


@pytest.fixture(scope="module")
def dg():
    import __graft_entry__
    __graft_entry__.build()
    import precision_matmul_dg_gb300 as dg
    assert torch.cuda.is_available()
    return dg


def _quantize_on_gpu(dg, x, K):
    """Runs dg_quantize_mxf4 into canary-filled buffers one row pitch (16
    bytes) and 3 scale bytes wider than needed; returns (codes [rows, K],
    scales [rows, nblk], raw code bytes, raw scale bytes)."""
    rows = x.shape[0]
    nblk = (K + 31) // 32
    ldq = (K + 31) // 32 * 32 + 32
    lds = nblk + 3
    X = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    Q = torch.full((rows, ldq // 2), CANARY, dtype=torch.uint8, device="cuda")
    S = torch.full((rows, lds), CANARY, dtype=torch.uint8, device="cuda")
    dg.quantize_mxf4_raw(rows, K, X, x.shape[1], Q, ldq, S, lds)
    dg.check_status()
    q, s = Q.cpu().numpy(), S.cpu().numpy()
    codes = oracle.gemm_ref.unpack_e2m1(q, K)
    return codes, s[:, :nblk], q, s


def _assert_quantize_parity(dg, x, K, rows=None):
    codes, scales, q, s = _quantize_on_gpu(dg, x, K)
    nblk = (K + 31) // 32
    sel = np.arange(x.shape[0]) if rows is None else rows
    ref_codes, ref_scales = oracle.mxfp4_quantize(x[sel], K)
    np.testing.assert_array_equal(scales[sel], ref_scales)
    bad = np.argwhere(codes[sel] != ref_codes)
    assert bad.size == 0, "%d code mismatches, first at %s: got %d want %d (x = %r)" % (
        len(bad), tuple(bad[0]), codes[sel][tuple(bad[0])], ref_codes[tuple(bad[0])],
        x[sel][bad[0][0], bad[0][1]])
    nbytes = (K + 1) // 2
    if K % 2:
        assert not (q[:, nbytes - 1] >> 4).any(), "high nibble past an odd K not zero"
    assert (q[:, nbytes:] == CANARY).all(), "codes written past the row"
    assert (s[:, nblk:] == CANARY).all(), "scales written past the row"


# ragged K (33, 1, 1000), and long rows (8200, 12296, 4104: more than one
# trip of a row's lanes, the last one short)
@pytest.mark.parametrize("shape", [(1, 32), (3, 40), (2, 33), (5, 1), (64, 1000), (257, 4096),
                                   (1000, 96), (7, 8), (9, 8200), (3, 12296), (5, 4104)],
                         ids=lambda s: "%dx%d" % s)
def test_quantize_parity(dg, shape):
    rows, K = shape
    x = workloads.mx_activations(rows, K, seed=rows * 7 + K)
    _assert_quantize_parity(dg, x, K)


def test_quantize_special_blocks(dg):
    K = 32 * 12
    x = workloads.mx_activations(6, K, seed=5)
    x[0, 3] = np.nan
    x[1, 40] = np.inf
    x[2, 70] = -np.inf
    x[3, 96:128] = 0.0
    x[4, 128:160] = np.float16(-0.0)
    # block 5 of row 5: amax 7.5 (X = 1) with every E2M1 tie, both signs
    ties = [4.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5, 7.5, 0.125, 1.0]
    x[5, 160:192] = 0.0
    x[5, 160:160 + len(ties)] = ties
    x[5, 176:176 + len(ties)] = [-t for t in ties]
    # block 6: FP16 subnormals only
    x[5, 192:224] = (np.arange(32) - 16).astype(np.float16) * np.float16(2.0 ** -24)
    # block 7: amax just below 2 (X = 1/4, amax / X just below 8: saturated)
    x[5, 224:256] = 0.01
    x[5, 224] = np.float16(2.0) - np.float16(2.0 ** -10)
    _assert_quantize_parity(dg, x, K)
    _, scales, _, _ = _quantize_on_gpu(dg, x, K)
    assert scales[0, 0] == 255 and scales[1, 1] == 255 and scales[2, 2] == 255
    assert scales[3, 3] == 0 and scales[4, 4] == 0


def test_quantize_full_size_sampled(dg):
    # the 4096 x 4096 activations of the square GEMM, rows sampled for the oracle
    x = workloads.mx_activations(4096, 4096, seed=11)
    rows = np.unique(np.concatenate([np.arange(0, 4096, 131), [4095]]))
    _assert_quantize_parity(dg, x, 4096, rows)


def _run_gemm(dg, case, plan=None):
    dev = "cuda"
    A = torch.from_numpy(case.A).to(dev)
    B = torch.from_numpy(case.B).to(dev)
    sa = torch.from_numpy(case.scale_a).to(dev)
    sb = torch.from_numpy(case.scale_b).to(dev)
    C = (torch.from_numpy(case.C).to(dev) if case.C is not None
         else torch.zeros(case.M, case.N, dtype=torch.float16, device=dev))
    bias = torch.from_numpy(case.bias).to(dev) if case.bias is not None else None
    dg.gemm_mxf4(A, sa, B, sb, C, case.K, bias=bias, alpha=case.alpha, beta=case.beta,
                 epilogue=case.epilogue, plan=plan)
    dg.check_status()
    return C.cpu().numpy()


def _assert_gemm_parity(case, got, rows=None):
    kw = dict(C=case.C, bias=case.bias, alpha=case.alpha, beta=case.beta,
              epilogue=case.epilogue, rows=rows)
    ref = oracle.gemm_mx_reference(case.A, case.scale_a, case.B, case.scale_b, case.K, **kw)
    bound = oracle.error_bound_mx(case.A, case.scale_a, case.B, case.scale_b, case.K, ref, **kw)
    g = (got if rows is None else got[rows]).astype(np.float64)
    nan_ref = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(g), nan_ref)
    err = np.abs(g - ref)
    ok = (err <= bound) | nan_ref
    if not ok.all():
        idx = tuple(np.argwhere(~ok)[0])
        raise AssertionError("%s: %d / %d outside the bound; first at %s: got %r want %r bound %r"
                             % (case.name, int((~ok).sum()), ok.size, idx, g[idx], ref[idx],
                                bound[idx]))


GEMM_CASES = [
    ((256, 520, 640), "none", 0.0),
    ((3, 300, 200), "bias_gelu", 0.5),          # M below one tile
    ((1, 8, 32), "none", 0.0),
    ((64, 64, 40), "bias", -1.0),               # ragged last block
    ((130, 1000, 1000), "gelu", 0.25),          # ragged K, ragged M
    ((1536, 2000, 512), "bias_gelu", 0.5),      # CTA-pair tiles
    ((1024, 2048, 1024), "none", 0.0),
]


@pytest.mark.parametrize("shape,epilogue,beta", GEMM_CASES,
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else str(v))
def test_gemm_mxf4_parity(dg, shape, epilogue, beta):
    M, N, K = shape
    case = workloads.mxf4_case(M, N, K, alpha=0.75, beta=beta, epilogue=epilogue,
                               seed=M + N + K)
    got = _run_gemm(dg, case)
    rows = None if M * N * K <= 2e9 else np.unique(np.concatenate([np.arange(0, M, 97), [M - 1]]))
    _assert_gemm_parity(case, got, rows)


def test_gemm_mxf4_wide_scale_range(dg):
    # A's block scales over 2^-67 .. 2^63 and B's all 2^-68: every value is
    # far outside FP16's range yet exact in BF16, and every product stays
    # below 2^-4 * 36, so D fits FP16 (products of the smallest blocks fall
    # below FP32's range, within the bound's 2^-24 floor)
    case = workloads.mxf4_case(200, 300, 256, seed=3, scale_lo=60, scale_hi=190)
    case.scale_b = np.full_like(case.scale_b, 59)
    _assert_gemm_parity(case, _run_gemm(dg, case))


def test_gemm_mxf4_nan_scale(dg):
    case = workloads.mxf4_case(64, 96, 128, seed=4)
    case.scale_a = case.scale_a.copy()
    case.scale_a[5, 1] = 255   # a NaN block in row 5 of A
    case.scale_b = case.scale_b.copy()
    case.scale_b[7, 3] = 255   # and one in column 7 of B
    got = _run_gemm(dg, case)
    assert np.isnan(got[5]).all() and np.isnan(got[:, 7]).all()
    _assert_gemm_parity(case, got)


def test_gemm_mxf4_k_zero(dg):
    case = workloads.mxf4_case(33, 70, 0, beta=0.5, epilogue="bias_gelu", seed=6)
    _assert_gemm_parity(case, _run_gemm(dg, case))


def test_gemm_mxf4_full_size_sampled(dg):
    # the bench configuration (4096^3, beta = 0.5) as bench.py runs it: the
    # FP16 activations quantized on the GPU, then the MXFP4 GEMM; the oracle
    # quantizes and multiplies a sample of the rows
    case = workloads.WORKLOADS["mxf4_4096"]()
    M, K = case.M, case.K
    Qa, Sa = dg.quantize_mxf4(torch.from_numpy(case.a_fp16).cuda(), K)
    C = torch.from_numpy(case.C).cuda()
    dg.gemm_mxf4(Qa, Sa, torch.from_numpy(case.B).cuda(), torch.from_numpy(case.scale_b).cuda(),
                 C, K, alpha=case.alpha, beta=case.beta, epilogue=case.epilogue)
    dg.check_status()
    rows = np.unique(np.concatenate([np.arange(0, M, 257), [M - 1]]))
    codes, scales = oracle.mxfp4_quantize(case.a_fp16[rows], K)
    np.testing.assert_array_equal(oracle.gemm_ref.unpack_e2m1(Qa.cpu().numpy()[rows], K), codes)
    np.testing.assert_array_equal(Sa.cpu().numpy()[rows], scales)
    sampled = workloads.Case(case.name, len(rows), case.N, K, "mxf4", "mxf4",
                             oracle.pack_e2m1(codes), case.B, case.C[rows], None, case.alpha,
                             case.beta, case.epilogue, scale_a=scales, scale_b=case.scale_b)
    _assert_gemm_parity(sampled, C.cpu().numpy()[rows])


def test_quantize_then_gemm(dg):
    # activations and weights quantized on the GPU, then multiplied: the
    # oracle quantizes the same FP16 rows and multiplies its own codes
    M, N, K = 96, 160, 300
    xa = workloads.mx_activations(M, K, seed=21, lo=-3, hi=3)
    xb = workloads.mx_activations(N, K, seed=22, lo=-3, hi=3)
    Qa, Sa = dg.quantize_mxf4(torch.from_numpy(xa).cuda(), K)
    Qb, Sb = dg.quantize_mxf4(torch.from_numpy(xb).cuda(), K)
    C = torch.zeros(M, N, dtype=torch.float16, device="cuda")
    dg.gemm_mxf4(Qa, Sa, Qb, Sb, C, K)
    dg.check_status()
    ca, sa = oracle.mxfp4_quantize(xa, K)
    cb, sb = oracle.mxfp4_quantize(xb, K)
    case = workloads.Case("quantized", M, N, K, "mxf4", "mxf4", oracle.pack_e2m1(ca),
                          oracle.pack_e2m1(cb), scale_a=sa, scale_b=sb)
    _assert_gemm_parity(case, C.cpu().numpy())


def test_quantize_padded_rows_not_read(dg):
    # X rows padded with NaN past K: a quantizer that read them would give
    # NaN scales (255) to the last blocks
    for K in (40, 100, 4096):
        x = workloads.mx_activations(9, K, seed=K)
        xp = np.full((9, (K + 7) // 8 * 8 + 24), np.nan, dtype=np.float16)
        xp[:, :K] = x[:, :K]
        _assert_quantize_parity(dg, xp, K)


@pytest.mark.parametrize("shape", [(70, 130, 100), (256, 300, 1024), (3, 40, 33)],
                         ids=lambda s: "x".join(map(str, s)))
def test_gemm_mxf4_padded_operands(dg, shape):
    # leading dimensions wider than the packed rows (the widening's general,
    # non-packed path): code padding holds random bytes, scale padding holds
    # NaN scales (255), so reading either would show in D
    M, N, K = shape
    case = workloads.mxf4_case(M, N, K, alpha=1.5, beta=0.5, epilogue="bias", seed=M * N + K)
    nblk = (K + 31) // 32
    rng = np.random.default_rng(7)

    def pad(codes, scales, extra_codes, extra_scales):
        rows = codes.shape[0]
        c = rng.integers(0, 256, (rows, codes.shape[1] + extra_codes // 2)).astype(np.uint8)
        c[:, :codes.shape[1]] = codes
        s = np.full((rows, nblk + extra_scales), 255, dtype=np.uint8)
        s[:, :nblk] = scales[:, :nblk]
        return c, s

    case.A, case.scale_a = pad(case.A, case.scale_a, 64, 5)
    case.B, case.scale_b = pad(case.B, case.scale_b, 32, 1)
    got = _run_gemm(dg, case)
    assert not np.isnan(got).any()
    _assert_gemm_parity(case, got)


@pytest.mark.parametrize("shape", [(256, 520, 640), (300, 460, 1000), (1, 100, 64),
                                   (520, 700, 512)],
                         ids=lambda s: "x".join(map(str, s)))
def test_gemm_mxf4_every_plan(dg, shape):
    # every plan the planner offers for the shape, the block-scaled MMA's
    # tiles (single CTAs: N_tile 224 and 128; CTA pairs: 256 x 224 and
    # 256 x 192) and the BF16 widening's, against the oracle (scale rows of
    # 20, 32, 2 and 16 bytes: copied to a 16-byte pitch first, or read by
    # TMA as they are)
    M, N, K = shape
    case = workloads.mxf4_case(M, N, K, alpha=1.25, beta=-0.5, epilogue="bias_gelu", seed=M + K)
    plans = dg.plan_tiles(M, N, K, "mxf4", "mxf4", max_out=64)
    native = {(p["n_tile"], p["stages"], p["cta_group"]) for p in plans
              if p["kernel_name"] == "tc"}
    want = {(224, 3, 1), (128, 5, 1)} | ({(224, 5, 2), (192, 5, 2)} if M > 128 else set())
    assert native == want
    for plan in plans:
        got = _run_gemm(dg, case, plan=plan)
        _assert_gemm_parity(case, got)


def test_gemm_mxf4_scale_layouts(dg):
    # the block-scaled kernel loads scale rows with TMA, which needs rows on
    # 16-byte boundaries: a padded pitch is read in place, a pitch or a base
    # off the boundary is copied to a 16-byte pitch first; all give the same
    # result, within the oracle's bound
    M, N, K = 300, 460, 1024
    case = workloads.mxf4_case(M, N, K, alpha=0.5, beta=0.25, epilogue="bias", seed=21)
    nblk = K // 32
    dev = "cuda"
    A = torch.from_numpy(case.A).to(dev)
    B = torch.from_numpy(case.B).to(dev)
    bias = torch.from_numpy(case.bias).to(dev)
    want = None
    for pad, off in ((0, 0), (16, 0), (48, 0), (16, 1), (5, 0), (8, 3)):
        sa_big = torch.full((M, nblk + pad + off), 7, dtype=torch.uint8, device=dev)
        sb_big = torch.full((N, nblk + pad + off), 7, dtype=torch.uint8, device=dev)
        sa = sa_big[:, off:off + nblk]
        sb = sb_big[:, off:off + nblk]
        sa.copy_(torch.from_numpy(case.scale_a))
        sb.copy_(torch.from_numpy(case.scale_b))
        C = torch.from_numpy(case.C).to(dev)
        plans = [p for p in dg.plan_tiles(M, N, K, "mxf4", "mxf4", max_out=64)
                 if p["kernel_name"] == "tc"]
        for plan in plans:
            C.copy_(torch.from_numpy(case.C))
            dg.gemm_mxf4(A, sa, B, sb, C, K, bias=bias, alpha=case.alpha, beta=case.beta,
                         epilogue=case.epilogue, plan=plan)
            dg.check_status()
            got = C.cpu().numpy()
            _assert_gemm_parity(case, got)
            if want is None:
                want = got
            else:  # one plan's tile order for every layout: the same bits
                if plan is plans[0]:
                    np.testing.assert_array_equal(got, want)


def test_gemm_mxf4_odd_k_is_widened(dg):
    # the block-scaled kernel reads whole bytes of codes: an odd K runs through
    # the widening, and a block-scaled plan is refused
    case = workloads.mxf4_case(64, 96, 99, beta=0.5, seed=9)
    plans = dg.plan_tiles(64, 96, 99, "mxf4", "mxf4", max_out=64)
    assert {p["kernel_name"] for p in plans} == {"tc_widened"}
    _assert_gemm_parity(case, _run_gemm(dg, case))
    native = dg.plan_tiles(64, 96, 100, "mxf4", "mxf4", max_out=64)
    native = next(p for p in native if p["kernel_name"] == "tc")
    with pytest.raises(dg.DgError) as ei:
        _run_gemm(dg, case, plan=native)
    assert ei.value.name == "DG_ERR_INVALID_STATE"
