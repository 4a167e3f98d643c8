"""Seeded synthetic inputs for the dg GEMM workloads.

This module only draws random numbers (a CPU torch.Generator, seed 0 by
default) and lays them out in the operand conventions of the library:
  A  M x K row-major (fp16 or int8),
  B  N rows of K (fp16 or int8), or N rows of K/2 bytes of packed 4-bit codes,
  C  M x N row-major (fp16),  bias  [N] (fp16).
It holds none of the GEMM arithmetic: the oracle and the CUDA path both take
their inputs from here and from nowhere else.

Random bytes are drawn uniformly over 0..255 for packed 4-bit weights, which
makes each of the two codes in a byte uniform over the 16 codes and
independent of the other, so no packing step is needed.
"""

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


@dataclass
class Case:
    name: str
    M: int
    N: int
    K: int
    dtype_a: str            # "f16" | "i8"
    dtype_b: str            # "f16" | "i8" | "e2m1"
    A: np.ndarray           # [M, lda]   (logical columns 0..K-1)
    B: np.ndarray           # [N, ldb] elements, or [N, ldb/2] bytes for e2m1
    C: Optional[np.ndarray] = None
    bias: Optional[np.ndarray] = None
    alpha: float = 1.0
    beta: float = 0.0
    epilogue: str = "none"
    lda: int = 0
    ldb: int = 0
    meta: dict = field(default_factory=dict)
    program: Optional[list] = None  # epilogue ops in order (replaces `epilogue`)
    batch: int = 1  # > 1: A [batch, M, lda], B [batch, N, ldb], C [batch, M, N]
    # dtype "mxf4": A [M, lda/2] and B [N, ldb/2] packed codes, with E8M0
    # scale bytes [M, ceil(K/32)] and [N, ceil(K/32)]
    scale_a: Optional[np.ndarray] = None
    scale_b: Optional[np.ndarray] = None
    # dtype "mxf4" with A given as FP16 activations [M, lda16] that the step
    # quantizes (A and scale_a are then None)
    a_fp16: Optional[np.ndarray] = None
    # a group of `batch` problems with their own row counts (A [batch, M, lda]
    # holds M = the largest count; problem g uses its first group_ms[g] rows)
    group_ms: Optional[list] = None

    def flops(self):
        if self.group_ms is not None:
            return 2.0 * sum(self.group_ms) * self.N * self.K
        return 2.0 * self.M * self.N * self.K * self.batch


def _gen(seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _normal(g, shape, std):
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.float16).numpy()


def _uniform_pm1(g, shape):
    x = torch.rand(*shape, generator=g, dtype=torch.float32)
    x.mul_(2.0).sub_(1.0)
    return x.to(torch.float16).numpy()


def _int8(g, shape):
    return torch.randint(-128, 128, shape, generator=g, dtype=torch.int16).to(torch.int8).numpy()


def _bytes(g, shape):
    return torch.randint(0, 256, shape, generator=g, dtype=torch.int16).to(torch.uint8).numpy()


def _pad_cols(x, ld, fill=0):
    """Place x [rows, cols] in a [rows, ld] buffer whose extra columns hold `fill`."""
    if ld == x.shape[1]:
        return np.ascontiguousarray(x)
    out = np.full((x.shape[0], ld), fill, dtype=x.dtype)
    out[:, : x.shape[1]] = x
    return out


def random_case(M, N, K, dtype_a="f16", dtype_b="f16", epilogue="none", alpha=1.0,
                beta=0.0, seed=0, dist="normal", lda=None, ldb=None, name=None, pad=0,
                program=None):
    """A general random case for parity tests.

    dist: "normal" -> N(0,1)/sqrt(K) operands (the square-GEMM recipe),
          "uniform" -> U[-1,1) operands.
    C ~ N(0,1) fp16 whenever beta != 0; bias ~ N(0, 0.1) fp16 when the
    epilogue (or the program) has a bias.  lda/ldb default to the smallest legal padded
    leading dimension (K rounded up to 8 fp16 / 16 int8 elements, 32 codes
    for packed 4-bit), so every leading dimension is a 16-byte multiple.
    pad: value stored in the columns between K and the leading dimension
    (e.g. NaN, to show those columns are never read).
    """
    g = _gen(seed)
    if dtype_a == "f16":
        lda = lda or _round_up(K, 8)
        if dist == "normal":
            A = _normal(g, (M, K), 1.0 / math.sqrt(K)) if dtype_b == "f16" else _normal(g, (M, K), 1.0)
        else:
            A = _uniform_pm1(g, (M, K))
    elif dtype_a == "i8":
        lda = lda or _round_up(K, 16)
        A = _int8(g, (M, K))
    else:
        raise ValueError(dtype_a)
    if dtype_b == "f16":
        ldb = ldb or _round_up(K, 8)
        B = _normal(g, (N, K), 1.0 / math.sqrt(K)) if dist == "normal" else _uniform_pm1(g, (N, K))
        B = _pad_cols(B, ldb, pad)
    elif dtype_b == "i8":
        ldb = ldb or _round_up(K, 16)
        B = _pad_cols(_int8(g, (N, K)), ldb, pad)
    elif dtype_b == "e2m1":
        ldb = ldb or _round_up(K, 32)
        nbytes = (K + 1) // 2
        Bp = _bytes(g, (N, nbytes))
        if K % 2:
            Bp[:, -1] &= 0x0F  # the unused high nibble of an odd row is left zero
        B = _pad_cols(Bp, ldb // 2, pad)
    else:
        raise ValueError(dtype_b)
    A = _pad_cols(A, lda, pad)
    C = None
    if beta != 0.0:
        C = _int32(g, (M, N)) if dtype_a == "i8" else _normal(g, (M, N), 1.0)
    bias = None
    if epilogue in ("bias", "bias_gelu") or any(
            op == "bias" or (isinstance(op, tuple) and op[0] == "bias") for op in program or []):
        bias = _normal(g, (N,), 0.1)
    return Case(name or "random_%s_%s_%dx%dx%d" % (dtype_a, dtype_b, M, N, K), M, N, K,
                dtype_a, dtype_b, A, B, C, bias, float(alpha), float(beta), epilogue, lda, ldb,
                program=list(program) if program else None)


def mxf4_case(M, N, K, alpha=1.0, beta=0.0, epilogue="none", seed=0, scale_lo=119,
              scale_hi=123, name=None, fp16_a=False):
    """MXFP4 operands drawn directly in their stored form: packed code bytes
    uniform over 0..255 (so every code of a row, including the ones past K in
    its last bytes, is uniform over the 16 E2M1 codes), and E8M0 scale bytes
    uniform over [scale_lo, scale_hi] (default 2^-8 .. 2^-4: the block scales
    of N(0,1)/sqrt(K) data at K of a few thousand); lda = ldb = K rounded up
    to 32 codes.  C ~ N(0,1) when beta != 0, bias ~ N(0, 0.1) for a bias
    epilogue.  With fp16_a, A is instead FP16 activations ~ N(0,1)/sqrt(K)
    (ld = K rounded up to 8) for the step to quantize."""
    g = _gen(seed)
    ld = _round_up(max(K, 1), 32)
    nblk = (K + 31) // 32
    A = _bytes(g, (M, ld // 2))
    B = _bytes(g, (N, ld // 2))
    sa = torch.randint(scale_lo, scale_hi + 1, (M, max(nblk, 1)), generator=g,
                       dtype=torch.int16).to(torch.uint8).numpy()
    sb = torch.randint(scale_lo, scale_hi + 1, (N, max(nblk, 1)), generator=g,
                       dtype=torch.int16).to(torch.uint8).numpy()
    C = _normal(g, (M, N), 1.0) if beta != 0.0 else None
    bias = _normal(g, (N,), 0.1) if epilogue in ("bias", "bias_gelu") else None
    a16 = None
    if fp16_a:
        a16 = _pad_cols(_normal(g, (M, K), 1.0 / math.sqrt(max(K, 1))), _round_up(max(K, 1), 8))
        A, sa = None, None
    return Case(name or "mxf4_%dx%dx%d" % (M, N, K), M, N, K, "mxf4", "mxf4", A, B, C, bias,
                float(alpha), float(beta), epilogue, ld, ld, scale_a=sa, scale_b=sb, a_fp16=a16)


def mx_activations(rows, K, seed=0, lo=-20, hi=12):
    """FP16 rows for block quantization: N(0,1) values times 2^e with e drawn
    per row uniformly in [lo, hi] (so the rows reach from FP16 subnormals to
    the thousands), ld = K rounded up to 8."""
    g = _gen(seed)
    x = torch.randn(rows, K, generator=g, dtype=torch.float32)
    e = torch.randint(lo, hi + 1, (rows, 1), generator=g, dtype=torch.int32).to(torch.float32)
    x = (x * torch.exp2(e)).to(torch.float16).numpy()
    return _pad_cols(x, _round_up(max(K, 1), 8))


def _int32(g, shape):
    return torch.randint(-(1 << 20), 1 << 20, shape, generator=g, dtype=torch.int32).numpy()


def _round_up(x, m):
    return (x + m - 1) // m * m


# ---------------------------------------------------------------------------
# The named workloads.  Each recipe states its sizes and distributions.
# ---------------------------------------------------------------------------

def f16_256(seed=0):
    """FP16 256^3, A and B ~ U[-1,1), alpha=1, beta=0, no epilogue."""
    c = random_case(256, 256, 256, "f16", "f16", dist="uniform", seed=seed, name="f16_256")
    return c


def f16_square(n, seed=0):
    """FP16 n^3, A,B ~ N(0,1)/sqrt(K), C ~ N(0,1), D = 1.0*A.B + 0.5*C."""
    return random_case(n, n, n, "f16", "f16", alpha=1.0, beta=0.5, seed=seed,
                       name="f16_%d" % n)


def f16_long_k(M, N, K, seed=0):
    """FP16 GEMM with fewer output tiles than the GPU has SMs and a long K (a
    projection of a few hundred rows), A,B ~ N(0,1)/sqrt(K), C ~ N(0,1),
    D = 1.0*A.B + 0.5*C."""
    return random_case(M, N, K, "f16", "f16", alpha=1.0, beta=0.5, seed=seed,
                       name="f16_%dx%dx%d" % (M, N, K))


def i8_square(n=4096, seed=0):
    """INT8 n^3, A,B uniform integers in [-128, 127], alpha=1, beta=0, int32 out."""
    return random_case(n, n, n, "i8", "i8", seed=seed, name="i8_%d" % n)


def thin(N, K, seed=0):
    """M=1 FP16 GEMV-shaped GEMM, a and B ~ N(0,1)/sqrt(K), alpha=1, beta=0."""
    return random_case(1, N, K, "f16", "f16", seed=seed, name="thin_1x%dx%d" % (N, K))


def w4a16(M, N=8960, K=1536, seed=0):
    """W4A16: packed E2M1 weights (uniform codes), A ~ N(0,1) fp16,
    bias ~ N(0, 0.1) fp16 (0.1 read as the standard deviation), bias + erf-GELU."""
    return random_case(M, N, K, "f16", "e2m1", epilogue="bias_gelu", seed=seed,
                       name="w4a16_m%d" % M)


def batched_thin(batch, N, K, seed=0):
    """`batch` independent M=1 FP16 GEMMs of one shape, e.g. the Q, K and V
    projections of 32 attention heads (96 problems of 1 x 128 x 4096); a and
    every B ~ N(0,1)/sqrt(K), alpha=1, beta=0."""
    g = _gen(seed)
    A = _normal(g, (batch, 1, K), 1.0 / math.sqrt(K))
    B = _normal(g, (batch, N, K), 1.0 / math.sqrt(K))
    return Case("qkv_1x%dx%d_b%d" % (N, K, batch), 1, N, K, "f16", "f16", A, B, lda=K, ldb=K,
                batch=batch)


def grouped_experts(count, N, K, m_hi=16, seed=0):
    """A mixture-of-experts layer: `count` experts with their own FP16
    weights B_g [N, K] ~ N(0,1)/sqrt(K) and row counts M_g uniform in
    [1, m_hi] (the tokens routed to each), activations ~ N(0,1)/sqrt(K),
    alpha=1, beta=0."""
    g = _gen(seed)
    ms = [int(x) for x in torch.randint(1, m_hi + 1, (count,), generator=g)]
    A = _normal(g, (count, m_hi, K), 1.0 / math.sqrt(K))
    B = _normal(g, (count, N, K), 1.0 / math.sqrt(K))
    return Case("moe_%dx%dx%d" % (count, N, K), m_hi, N, K, "f16", "f16", A, B, lda=K, ldb=K,
                batch=count, group_ms=ms)


WORKLOADS = {
    "f16_256": lambda: f16_256(),
    "f16_2048": lambda: f16_square(2048),
    "f16_4096": lambda: f16_square(4096),
    "f16_8192": lambda: f16_square(8192),
    "f16_256x4096x16384": lambda: f16_long_k(256, 4096, 16384),
    "i8_4096": lambda: i8_square(4096),
    "thin_1x4096x131072": lambda: thin(4096, 131072),
    "thin_1x256x12800": lambda: thin(256, 12800),
    "w4a16_m16": lambda: w4a16(16),
    "w4a16_m256": lambda: w4a16(256),
    "w4a16_m2048": lambda: w4a16(2048),
    "qkv_1x128x4096_b96": lambda: batched_thin(96, 128, 4096),
    "mxf4_4096": lambda: mxf4_case(4096, 4096, 4096, beta=0.5, name="mxf4_4096", fp16_a=True),
    "moe_64x4096x2048": lambda: grouped_experts(64, 4096, 2048),
}
