"""CPU oracle for the dg GEMM path -- TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously-correct definition of what the
library computes.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it.  The product path (the CUDA
library and its Python binding) never imports, links or calls anything here,
and nothing here imports the product path.

Sources (cited by page address and section):
  * discosf.com/news/5532976 -- "DeepGEMM" article, section 2.2 layer 2
    (weight int4_e2m1 / activation fp16 / output fp16 precision triple),
    section 3.5 experience 2 (FP32 accumulation, cast_output fp16),
    section 4.1 stage 4 (correctness proposition |C - A x B| <= eps),
    section 4.3 (packed 4-bit weights), section 6.1 (GELU fused epilogue).
  * kwkr.cn/news/562171 -- "DeepGEMM" article, section 2.2 third layer
    (epilogue generator: alpha * gemm_out + beta * ..., bias + GELU fused),
    section 3.2 step 3 (epilogue "alpha * C + beta * D").

Block-scaled 4-bit operands (MXFP4: E2M1 codes with one E8M0 scale per 32
values along K) and the GEMM on them are in ``oracle.mx_ref``; the pages fix
no block format, and that module's docstring states the reading taken.

Parity status of each function is listed in ``oracle.gemm_ref.__doc__`` and
``oracle.mx_ref.__doc__``.
"""

from .gemm_ref import (  # noqa: F401
    E2M1_BITS,
    e2m1_value,
    e2m1_decode,
    unpack_e2m1,
    gelu_erf,
    gemm_reference,
    error_bound,
    apply_program,
    quantize_i8,
    PROGRAM_OPS,
    GELU_LIPSCHITZ,
)
from .mx_ref import (  # noqa: F401
    MX_BLOCK,
    e8m0_value,
    e8m0_decode,
    e2m1_round,
    shared_exponent,
    mxfp4_quantize,
    mxfp4_dequantize,
    pack_e2m1,
    gemm_mx_reference,
    error_bound_mx,
)
