"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Floating point: every element within 2^-10 * (|A|.|B|)_ij + 2^-10 * |D_ref|_ij
(plus the 2^-24 floor and the GELU factor, see oracle.error_bound).
INT8: bit-exact.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import assert_parity, run_case, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    import __graft_entry__
    __graft_entry__.build()
    import precision_matmul_dg_gb300 as dg
    assert torch.cuda.is_available()
    return dg


# ------------------------------------------------------- full-size workloads
@pytest.mark.parametrize("name", ["f16_256", "f16_2048", "f16_4096", "f16_8192",
                                  "f16_256x4096x16384", "thin_1x256x12800",
                                  "thin_1x4096x131072"])
def test_workload_full_size(dg, name):
    case = workloads.WORKLOADS[name]()
    got, _ = run_case(dg, case)
    assert_parity(case, got)


# ------------------------------------------------------- shapes and tails
RANDOM = [
    (128, 256, 64), (300, 520, 200), (129, 257, 72), (1000, 17, 99), (17, 1000, 130),
    (512, 384, 1000), (640, 768, 4096), (77, 2000, 333), (1031, 263, 1),
]


@pytest.mark.parametrize("shape", RANDOM, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("epi", ["none", "bias", "gelu", "bias_gelu"])
def test_random_shapes(dg, shape, epi):
    M, N, K = shape
    case = workloads.random_case(M, N, K, epilogue=epi, alpha=-0.75, beta=0.5,
                                 seed=hash((M, N, K, epi)) % 1000, pad=float("nan"))
    got, _ = run_case(dg, case)
    assert_parity(case, got)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("K", [8, 100, 256, 4097, 20000])
def test_thin_m(dg, M, K):
    case = workloads.random_case(M, 300, K, epilogue="bias", beta=-1.25, seed=M * 7 + K,
                                 pad=float("nan"))
    got, _ = run_case(dg, case)
    assert_parity(case, got)


def _plans(dg, case):
    return dg.plan_tiles(case.M, case.N, case.K, case.dtype_a, case.dtype_b, case.epilogue,
                         target_occupancy=0.0)


def test_every_tensor_core_plan(dg):
    case = workloads.random_case(520, 1100, 700, epilogue="bias_gelu", alpha=1.5, beta=0.25,
                                 seed=5)
    tc = [p for p in _plans(dg, case) if p["kernel_name"] == "tc"]
    assert {p["n_tile"] for p in tc} == {64, 128, 192, 224, 256}
    for p in tc:
        for grid in (p["grid"], 7, 1):   # persistent CTAs walking several tiles each
            q = dict(p, grid=grid)
            got, _ = run_case(dg, case, plan=q)
            assert_parity(case, got)


def test_every_gemv_split(dg):
    case = workloads.random_case(3, 200, 30000, beta=0.5, epilogue="gelu", seed=9)
    gv = [p for p in _plans(dg, case) if p["kernel_name"] == "gemv"]
    assert {p["split_k"] for p in gv} >= {1, 2, 4, 8}
    outs = []
    for p in gv:
        got, _ = run_case(dg, case, plan=p)
        assert_parity(case, got)
        outs.append(got)


@pytest.mark.parametrize("M", [2, 7, 8, 9, 15, 16])
@pytest.mark.parametrize("K", [1, 8, 31, 100, 4097, 20000])
def test_gemv_mma(dg, M, K):
    # warp-MMA GEMV: ragged N (not a multiple of the 64-column CTA), K tails
    # shorter than one 32-wide step, padding columns holding NaN
    case = workloads.random_case(M, 300, K, epilogue="bias_gelu", alpha=0.75, beta=-1.25,
                                 seed=M * 31 + K, pad=float("nan"))
    plan = [p for p in _plans(dg, case) if p["kernel_name"] == "gemv_mma"][0]
    got, _ = run_case(dg, case, plan=plan)
    assert_parity(case, got)


def test_every_gemv_mma_split(dg):
    case = workloads.random_case(12, 200, 30000, beta=0.5, epilogue="gelu", seed=19)
    gm = [p for p in _plans(dg, case) if p["kernel_name"] == "gemv_mma"]
    assert {p["split_k"] for p in gm} >= {1, 2, 4, 8, 14}
    for p in gm:
        got, _ = run_case(dg, case, plan=p)
        assert_parity(case, got)


# ------------------------------------------------------- edge cases
def test_k_zero(dg):
    for epi in ("none", "bias_gelu"):
        case = workloads.random_case(33, 70, 8, epilogue=epi, beta=0.5, seed=3)
        case.K = 0
        got, _ = run_case(dg, case)
        assert_parity(case, got)


def test_empty_m_or_n(dg):
    A = torch.zeros(4, 8, dtype=torch.float16, device="cuda")
    B = torch.zeros(4, 8, dtype=torch.float16, device="cuda")
    C = torch.zeros(0, 4, dtype=torch.float16, device="cuda")
    before = dg.launch_count()
    dg.gemm_raw(0, 4, 8, "f16", "f16", A, 8, B, 8, A, None, 1.0, 0.0, "none")
    dg.gemm_raw(4, 0, 8, "f16", "f16", A, 8, B, 8, A, None, 1.0, 0.0, "none")
    assert dg.launch_count() == before
    del C


def test_output_canary_untouched(dg):
    for shape in [(129, 257, 72), (1, 1000, 5000), (256, 256, 256), (5, 3, 17)]:
        case = workloads.random_case(*shape, epilogue="gelu", beta=0.5, seed=1)
        got, tail = run_case(dg, case, canary=64)
        assert_parity(case, got)
        assert np.all(tail == np.float16(-7.5))


def _run_at_offset(dg, case, off, guard=64, plan=None):
    """Runs `case` with C/D placed `off` elements into a larger buffer whose
    `guard` elements before and after are filled with a canary."""
    n = case.M * case.N
    buf = torch.full((off + n + guard,), -7.5, dtype=torch.float16, device="cuda")
    A, B, C0, bias, _ = to_device(case)
    C = buf[off:off + n].view(case.M, case.N)
    C.copy_(C0)
    dg.gemm(A, B, C, K=case.K, bias=bias, alpha=case.alpha, beta=case.beta,
            epilogue=case.epilogue, plan=plan)
    dg.check_status()
    host = buf.cpu().numpy()
    assert np.all(host[:off] == np.float16(-7.5)) and np.all(host[off + n:] == np.float16(-7.5))
    return C.cpu().numpy()


@pytest.mark.parametrize("shape", [(300, 520, 200), (256, 1000, 640), (129, 72, 1000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_staged_epilogue_at_offset(dg, shape):
    # D 16 bytes into a larger buffer (aligned for TMA, not to a line): the
    # boxes write exactly the M x N elements, none of the guards around them.
    case = workloads.random_case(*shape, epilogue="bias_gelu", alpha=0.75, beta=-0.5, seed=11)
    got = _run_at_offset(dg, case, 8)
    assert_parity(case, got)


def test_every_tensor_core_plan_without_c(dg):
    # beta = 0: the staged epilogue stores only (no C loads)
    case = workloads.random_case(700, 904, 520, epilogue="bias_gelu", alpha=-1.25, seed=12)
    for p in [p for p in _plans(dg, case) if p["kernel_name"] == "tc"]:
        got, tail = run_case(dg, case, plan=p, canary=64)
        assert_parity(case, got)
        assert np.all(tail == np.float16(-7.5))


def test_padded_leading_dimensions(dg):
    case = workloads.random_case(200, 300, 100, lda=160, ldb=136, beta=0.5, seed=4,
                                 pad=float("nan"))
    got, _ = run_case(dg, case)
    assert_parity(case, got)


def test_deterministic(dg):
    for shape in [(1000, 1000, 1000), (1, 4096, 65536)]:
        case = workloads.random_case(*shape, beta=0.5, seed=2)
        a, _ = run_case(dg, case)
        b, _ = run_case(dg, case)
        assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_closed_forms_on_device(dg):
    # all-ones: D = K exactly;  identity B: D = A exactly
    K = 4096
    case = workloads.random_case(256, 256, K, seed=0)
    case.A = np.ones_like(case.A)
    case.B = np.ones_like(case.B)
    got, _ = run_case(dg, case)
    assert np.all(got == np.float16(K))
    case = workloads.random_case(300, 192, 192, seed=6)
    case.B = np.eye(192, dtype=np.float16)
    got, _ = run_case(dg, case)
    assert np.array_equal(got, case.A[:, :192])


def test_back_to_back_kernels_keep_stream_order(dg):
    # Tensor-core launches overlap the previous kernel's drain (programmatic
    # dependent launch) and wait for it before touching global memory.  Three
    # launches with no host synchronisation: step 2 reads step 1's output
    # (read after write) and overwrites step 1's input (write after read);
    # step 3 reads step 2's output and updates its own C in place.
    M, K = 640, 1024
    base = [workloads.random_case(M, K, K, seed=31 + i) for i in range(3)]
    P0 = base[0].A.copy()
    R0 = np.random.default_rng(7).standard_normal((M, K)).astype(np.float16)
    dev = "cuda:0"
    P = torch.from_numpy(P0).to(dev)
    Q = torch.zeros(M, K, dtype=torch.float16, device=dev)
    R = torch.from_numpy(R0).to(dev)
    W = [torch.from_numpy(c.B).to(dev) for c in base]
    for _ in range(3):   # repeated, so later launches also overlap earlier ones
        P.copy_(torch.from_numpy(P0).to(dev))
        R.copy_(torch.from_numpy(R0).to(dev))
        dg.gemm(P, W[0], Q)                   # Q = P . W0^T
        dg.gemm(Q, W[1], P)                   # P = Q . W1^T
        dg.gemm(P, W[2], R, beta=0.5)         # R = P . W2^T + 0.5 R
    dg.check_status()
    q, p, r = Q.cpu().numpy(), P.cpu().numpy(), R.cpu().numpy()
    steps = [(P0, q, None, 0.0), (q, p, None, 0.0), (p, r, R0, 0.5)]
    for (a, got, c, beta), cs in zip(steps, base):
        cs.A, cs.C, cs.beta = a, c, beta
        assert_parity(cs, got)


def test_back_to_back_widened_and_gemv_keep_stream_order(dg):
    # Every kernel of the library is launched as a programmatic dependent.
    # (1) Two widened INT8 GEMMs with no host synchronisation: the second one's
    # widening pass overwrites the FP16 workspace the first one's tensor-core
    # kernel reads (write after read).  (2) Thin GEMV launches each reading
    # the previous one's output (read after write).
    dev = "cuda:0"
    cases = [workloads.random_case(640, 1024, 1024, "i8", "i8", seed=41 + i) for i in range(2)]
    plan = [p for p in _plans(dg, cases[0]) if p["kernel_name"] == "tc_widened"][0]
    outs = []
    for _ in range(2):
        outs = []
        for cs in cases:
            A = torch.from_numpy(cs.A).to(dev)
            B = torch.from_numpy(cs.B).to(dev)
            C = torch.zeros(cs.M, cs.N, dtype=torch.int32, device=dev)
            dg.gemm(A, B, C, plan=plan)
            outs.append(C)
    dg.check_status()
    for cs, C in zip(cases, outs):
        assert_parity(cs, C.cpu().numpy())
    K = 2048
    chain = [workloads.random_case(2, K, K, seed=51 + i) for i in range(3)]
    x0 = chain[0].A.copy()
    X = [torch.from_numpy(x0).to(dev)] + [torch.zeros(2, K, dtype=torch.float16, device=dev)
                                          for _ in chain]
    W = [torch.from_numpy(c.B).to(dev) for c in chain]
    for i in range(len(chain)):
        dg.gemm(X[i], W[i], X[i + 1])          # X[i+1] = X[i] . W[i]^T
    dg.check_status()
    host = [x.cpu().numpy() for x in X]
    for i, cs in enumerate(chain):
        cs.A = host[i]
        assert_parity(cs, host[i + 1])


@pytest.mark.parametrize("m", [4096, 5])   # tensor-core kernel, thin GEMV
def test_gelu_grid(dg, m):
    # K = 1, B = 1: D = GELU(x) for a grid of FP16 x over [-12, 12].
    case = workloads.random_case(m, 64, 1, epilogue="gelu", seed=3)
    x = np.linspace(-12.0, 12.0, m).astype(np.float16)
    case.A = np.zeros_like(case.A)
    case.A[:, 0] = x
    case.B = np.zeros_like(case.B)
    case.B[:, 0] = 1.0
    got, _ = run_case(dg, case)
    assert_parity(case, got)
    # where Phi(x) is not tiny the result is the correctly rounded FP16 value
    # or a neighbour (the FP32 arithmetic carries ~1e-7 relative error)
    ref = np.float16(oracle.gelu_erf(x.astype(np.float64)))
    sel = x >= -2.0
    ulp = np.abs(np.spacing(ref[sel]).astype(np.float64))
    diff = np.abs(got[sel, 0].astype(np.float64) - ref[sel].astype(np.float64))
    assert np.all(diff <= ulp)


def test_side_stream(dg):
    s = torch.cuda.Stream()
    case = workloads.random_case(384, 640, 512, epilogue="bias", beta=0.5, seed=8)
    with torch.cuda.stream(s):
        got, _ = run_case(dg, case, stream=s)
    assert_parity(case, got)


def test_timeout_is_reported_and_context_survives(dg):
    dg.set_wait_timeout_ns(2_000_000)  # 2 ms
    try:
        dg.selftest_wait_timeout()
        with pytest.raises(dg.DgError) as ei:
            dg.check_status()
        assert ei.value.name == "DG_ERR_TIMEOUT"
    finally:
        dg.set_wait_timeout_ns(0)
    dg.check_status()  # cleared
    case = workloads.random_case(256, 256, 256, seed=1)
    got, _ = run_case(dg, case)
    assert_parity(case, got)


# ------------------------------------------------------- INT8 (bit-exact)
@pytest.mark.parametrize("name", ["i8_4096"])
def test_int8_workload_full_size(dg, name):
    case = workloads.WORKLOADS[name]()
    got, _ = run_case(dg, case)
    assert_parity(case, got)


@pytest.mark.parametrize("shape", [(128, 128, 64), (300, 520, 200), (129, 257, 72),
                                   (1000, 17, 99), (17, 1000, 1030), (256, 384, 2049),
                                   (640, 768, 4096), (7, 9, 5), (1031, 263, 1)],
                         ids=lambda s: "x".join(map(str, s)))
def test_int8_random_shapes(dg, shape):
    M, N, K = shape
    case = workloads.random_case(M, N, K, "i8", "i8", alpha=3, beta=-2, seed=M + N + K, pad=127)
    got, _ = run_case(dg, case)
    assert_parity(case, got)


def test_int8_extremes_and_wraparound(dg):
    K = 4096
    for a_val, b_val in [(-128, -128), (127, -128), (-128, 127), (127, 127)]:
        case = workloads.random_case(130, 260, K, "i8", "i8", seed=1)
        case.A = np.full_like(case.A, a_val)
        case.B = np.full_like(case.B, b_val)
        got, _ = run_case(dg, case)
        assert np.all(got == a_val * b_val * K)
    # alpha large enough to wrap modulo 2^32
    case = workloads.random_case(64, 96, 3000, "i8", "i8", alpha=65537, beta=7, seed=2)
    got, _ = run_case(dg, case)
    assert_parity(case, got)


def test_int8_every_plan(dg):
    # converting kernel and widened plans (1 CTA and CTA pair, exact INT32 mode);
    # K = 2500 spans three exact-FP32 chunks of 1024 and a ragged tail
    case = workloads.random_case(300, 600, 2500, "i8", "i8", alpha=1, beta=1, seed=3)
    plans = [p for p in _plans(dg, case) if p["kernel_name"] in ("tc", "tc_widened")]
    assert {p["kernel_name"] for p in plans} == {"tc", "tc_widened"}
    assert {p["cta_group"] for p in plans} == {1, 2}
    for p in plans:
        for grid in (p["grid"], 3):
            got, _ = run_case(dg, case, plan=dict(p, grid=grid))
            assert_parity(case, got)
    # N % 4 != 0: INT32 rows are not 16-byte multiples, D is stored from registers
    case = workloads.random_case(300, 603, 1100, "i8", "i8", alpha=-3, beta=-2, seed=4)
    for p in _plans(dg, case):
        if p["kernel_name"] == "tc_widened":
            got, _ = run_case(dg, case, plan=p)
            assert_parity(case, got)


def test_int8_widened_extremes(dg):
    # adversarial exactness through the widened path: all -128 (chunk sums of
    # exactly 2^24) and mixed extremes, at sizes where the planner widens
    K = 4096
    for a_val, b_val in [(-128, -128), (127, -128)]:
        case = workloads.random_case(512, 512, K, "i8", "i8", seed=1)
        case.A = np.full_like(case.A, a_val)
        case.B = np.full_like(case.B, b_val)
        for p in _plans(dg, case):
            if p["kernel_name"] == "tc_widened":
                got, _ = run_case(dg, case, plan=p)
                assert np.all(got == a_val * b_val * K), p


# ------------------------------------------------------- W4A16
@pytest.mark.parametrize("name", ["w4a16_m16", "w4a16_m256", "w4a16_m2048"])
def test_w4a16_workload_full_size(dg, name):
    case = workloads.WORKLOADS[name]()
    got, _ = run_case(dg, case)
    assert_parity(case, got)


@pytest.mark.parametrize("shape", [(16, 8960, 1536), (300, 520, 200), (129, 257, 71),
                                   (1000, 17, 99), (5, 1000, 1030), (640, 768, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("epi", ["none", "bias_gelu"])
def test_w4a16_random_shapes(dg, shape, epi):
    M, N, K = shape
    case = workloads.random_case(M, N, K, "f16", "e2m1", epilogue=epi, alpha=0.5, beta=0.25,
                                 seed=M * 3 + K, pad=255)
    got, _ = run_case(dg, case)
    assert_parity(case, got)


def _skinny_plan(dg, case):
    sk = [p for p in _plans(dg, case) if p["kernel_name"] == "skinny"]
    assert len(sk) == 1
    return sk[0]


@pytest.mark.parametrize("shape", [(16, 8960, 1536), (1, 100, 64), (3, 777, 33), (9, 130, 4100),
                                   (16, 64, 2048), (13, 1001, 6000), (2, 65, 1)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("epi", ["none", "bias_gelu"])
def test_w4a16_skinny(dg, shape, epi):
    # warp-MMA skinny kernel (M <= 16): ragged N (partial 64-column blocks and
    # 8-column groups), K tails inside a 32-code group and across 2048-code
    # chunks; the padding bytes (0xFF codes) past K must not contribute
    M, N, K = shape
    case = workloads.random_case(M, N, K, "f16", "e2m1", epilogue=epi, alpha=-0.75, beta=0.5,
                                 seed=M * 7 + N + K, pad=255)
    got, tail = run_case(dg, case, plan=_skinny_plan(dg, case), canary=64)
    assert_parity(case, got)
    assert np.all(tail == np.float16(-7.5))


def test_w4a16_skinny_every_m(dg):
    # every row count 1..16 through the same column layout
    for M in range(1, 17):
        case = workloads.random_case(M, 200, 700, "f16", "e2m1", epilogue="bias", beta=-1.0,
                                     seed=100 + M, pad=255)
        got, _ = run_case(dg, case, plan=_skinny_plan(dg, case))
        assert_parity(case, got)


def test_w4a16_every_code_one_hot(dg):
    """Column j of the weights holds code j % 16 at k = j % K and zeros elsewhere,
    so D[:, j] = A[:, k] * value(code): every code's decoded value appears as a
    product with an exact fp16 activation (table from the pinned golden file)."""
    table = {}
    import os
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "e2m1_codes.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            c, v = line.split()
            table[int(c)] = float(v)
    M, N, K = 64, 64, 64
    case = workloads.random_case(M, N, K, "f16", "e2m1", seed=4)
    case.A = np.ascontiguousarray(np.round(case.A * 8) / 8).astype(np.float16)
    packed = np.zeros_like(case.B)
    for j in range(N):
        k, code = j % K, j % 16
        packed[j, k // 2] |= np.uint8(code << (4 * (k % 2)))
    case.B = packed
    got, _ = run_case(dg, case)
    for j in range(N):
        want = case.A[:, j % K].astype(np.float64) * table[j % 16]
        assert np.array_equal(got[:, j].astype(np.float64), want), j


def test_w4a16_every_plan(dg):
    case = workloads.random_case(200, 700, 600, "f16", "e2m1", epilogue="bias_gelu", beta=0.5,
                                 seed=5)
    plans = [p for p in _plans(dg, case) if p["kernel_name"] in ("tc", "tc_widened")]
    assert {p["n_tile"] for p in plans if p["kernel_name"] == "tc" and not p["swap_ab"]} == \
        {64, 128, 256}
    assert {p["n_tile"] for p in plans if p["kernel_name"] == "tc" and p["swap_ab"]} == {160, 224}
    assert {p["n_tile"] for p in plans if p["kernel_name"] == "tc_widened"} >= {128, 224, 256}
    assert {p["cta_group"] for p in plans if p["kernel_name"] == "tc_widened"} == {1, 2}
    for p in plans:
        got, _ = run_case(dg, case, plan=p)
        assert_parity(case, got)


# ------------------------------------------------------- host-buffer entry point
def _run_host(dg, case, pinned=True, in_place=False, stream=None):
    def host(x):
        t = torch.from_numpy(np.array(x, copy=True))  # never alias the case's own arrays
        return t.pin_memory() if pinned else t
    A, B = host(case.A), host(case.B)
    out_dtype = torch.int32 if case.dtype_a == "i8" else torch.float16
    C = host(case.C) if case.C is not None else None
    if in_place:
        assert C is not None
        D = C
    else:
        D = torch.full((case.M, case.N), 3, dtype=out_dtype)
        D = D.pin_memory() if pinned else D
    bias = host(case.bias) if case.bias is not None else None
    dg.gemm_host(A, B, D, C=C, K=case.K, bias=bias, alpha=case.alpha, beta=case.beta,
                 epilogue=case.epilogue, dtype_b=case.dtype_b, stream=stream)
    torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
    dg.check_status()
    return D.numpy().copy()


@pytest.mark.parametrize("spec", [
    ("f16", "f16", (1100, 700, 900), "bias_gelu", 0.5),     # tensor cores, 3 row panels
    ("f16", "f16", (4096, 4096, 4096), "none", 0.5),        # the square workload
    ("f16", "f16", (5, 3000, 2000), "bias", -1.0),          # thin GEMV
    ("i8", "i8", (600, 520, 700), "none", 2.0),             # exact INT32
    ("f16", "e2m1", (16, 900, 1536), "bias_gelu", 0.0),     # skinny
    ("f16", "e2m1", (520, 1000, 400), "gelu", 0.25),        # converting / widened
], ids=lambda s: "%s_%s_%dx%dx%d_%s" % (s[0], s[1], *s[2], s[3]))
def test_gemm_host(dg, spec):
    da, db, (M, N, K), epi, beta = spec
    case = workloads.random_case(M, N, K, da, db, epilogue=epi, beta=beta,
                                 alpha=1 if da == "i8" else 0.75, seed=M + N + K, pad=0)
    got = _run_host(dg, case)
    assert_parity(case, got)


def test_gemm_host_pageable_in_place_and_reuse(dg):
    # pageable host memory; D == C; shapes that grow and shrink the workspace;
    # back-to-back calls on one stream with no synchronisation between them
    cases = [workloads.random_case(300, 256, 512, epilogue="bias", beta=0.5, seed=61),
             workloads.random_case(1500, 520, 640, beta=-0.5, seed=62),
             workloads.random_case(40, 100, 64, epilogue="gelu", beta=1.0, seed=63)]
    for cs in cases:
        assert_parity(cs, _run_host(dg, cs, pinned=False, in_place=True))
    s = torch.cuda.Stream()
    outs = []
    hosts = []
    for cs in cases:
        A = torch.from_numpy(cs.A).pin_memory()
        B = torch.from_numpy(cs.B).pin_memory()
        C = torch.from_numpy(cs.C).pin_memory()
        D = torch.empty(cs.M, cs.N, dtype=torch.float16).pin_memory()
        bias = torch.from_numpy(cs.bias).pin_memory() if cs.bias is not None else None
        dg.gemm_host(A, B, D, C=C, bias=bias, alpha=cs.alpha, beta=cs.beta,
                     epilogue=cs.epilogue, stream=s)
        hosts.append((A, B, C, bias))
        outs.append(D)
    s.synchronize()
    dg.check_status(s)
    for cs, D in zip(cases, outs):
        assert_parity(cs, D.numpy())
