"""Host-side checks of the C ABI: the library builds and loads, exports every
symbol include/dg.h declares, its struct layouts match the binding, and
invalid arguments are rejected synchronously (no GPU needed)."""

import ctypes
import os
import re
import subprocess
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dg.h")


@pytest.fixture(scope="module")
def dg():
    import __graft_entry__
    __graft_entry__.build()
    import precision_matmul_dg_gb300 as dg
    return dg


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_exports(dg):
    assert _declared_functions() == sorted(dg.EXPORTS)


def test_library_exports_every_declared_symbol(dg):
    L = ctypes.CDLL(dg.lib_path())
    for name in _declared_functions():
        assert hasattr(L, name), name
    nm = subprocess.run(["nm", "-D", "--defined-only", dg.lib_path()], capture_output=True,
                        text=True)
    if nm.returncode == 0:
        defined = set(re.findall(r"\s[TW]\s+(\S+)", nm.stdout))
        for name in _declared_functions():
            assert name in defined, name


def test_struct_layout_matches_c(dg, tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(textwrap.dedent("""
        #include <stdio.h>
        #include <stddef.h>
        #include "dg.h"
        #define F(T, f) printf(#T "." #f " %zu\\n", offsetof(T, f));
        int main(void) {
          printf("dg_hw_desc %zu\\n", sizeof(dg_hw_desc));
          printf("dg_tile_plan %zu\\n", sizeof(dg_tile_plan));
          printf("dg_epilogue_op %zu\\n", sizeof(dg_epilogue_op));
          printf("dg_epilogue_program %zu\\n", sizeof(dg_epilogue_program));
          printf("ops %d,%d,%d,%d,%d,%d\\n", DG_MAX_EPILOGUE_OPS, DG_OP_BIAS, DG_OP_RELU,
                 DG_OP_GELU, DG_OP_SCALE, DG_OP_CLAMP);
          printf("dtypes %d,%d,%d,%d\\n", DG_F16, DG_I8, DG_E2M1, DG_MXF4);
          printf("kernels %d,%d,%d,%d,%d\\n", DG_KERNEL_TC, DG_KERNEL_GEMV, DG_KERNEL_TC_WIDENED,
                 DG_KERNEL_SKINNY, DG_KERNEL_GEMV_MMA);
          F(dg_hw_desc, l2_bytes) F(dg_hw_desc, hbm_gbps) F(dg_hw_desc, clock_ghz)
          F(dg_tile_plan, regs_per_thread) F(dg_tile_plan, grid) F(dg_tile_plan, occupancy) F(dg_tile_plan, est_tflops)
          F(dg_epilogue_op, a) F(dg_epilogue_op, b) F(dg_epilogue_program, ops)
          return 0;
        }
    """))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    out = dict(line.rsplit(" ", 1) for line in subprocess.run(
        [str(exe)], capture_output=True, text=True, check=True).stdout.split("\n") if line)
    assert int(out["dg_hw_desc"]) == ctypes.sizeof(dg.HwDesc)
    assert int(out["dg_tile_plan"]) == ctypes.sizeof(dg.TilePlan)
    assert int(out["dg_epilogue_op"]) == ctypes.sizeof(dg.EpilogueOp)
    assert int(out["dg_epilogue_program"]) == ctypes.sizeof(dg.EpilogueProgram)
    ops = [int(x) for x in out.pop("ops").split(",")]
    assert [int(x) for x in out.pop("dtypes").split(",")] == [dg.DTYPES[k] for k in
                                                              ("f16", "i8", "e2m1", "mxf4")]
    kernels = [int(x) for x in out.pop("kernels").split(",")]
    assert [dg.KERNELS[k] for k in kernels] == ["tc", "gemv", "tc_widened", "skinny", "gemv_mma"]
    assert ops == [dg.MAX_EPILOGUE_OPS] + [dg.OPS[k] for k in ("bias", "relu", "gelu", "scale",
                                                               "clamp")]
    classes = {"dg_hw_desc": dg.HwDesc, "dg_tile_plan": dg.TilePlan,
               "dg_epilogue_op": dg.EpilogueOp, "dg_epilogue_program": dg.EpilogueProgram}
    for key, val in out.items():
        if "." in key:
            struct, field = key.split(".")
            assert getattr(classes[struct], field).offset == int(val), key


# ---------------------------------------------------------------- validation
# Pointers below are fake device addresses: every call must be rejected (or be
# a no-op) before anything touches a GPU.

GOOD = dict(M=64, N=64, K=64, dtype_a="f16", dtype_b="f16", A=0x10000, lda=64, B=0x20000, ldb=64,
            C=0x30000, bias=None, alpha=1.0, beta=0.0, epilogue="none")


def _call(dg, **over):
    kw = dict(GOOD)
    kw.update(over)
    try:
        dg.gemm_raw(kw["M"], kw["N"], kw["K"], kw["dtype_a"], kw["dtype_b"], kw["A"], kw["lda"],
                    kw["B"], kw["ldb"], kw["C"], kw["bias"], kw["alpha"], kw["beta"],
                    kw["epilogue"], stream=0)
    except dg.DgError as e:
        return e.name, str(e)
    return "DG_OK", ""


@pytest.mark.parametrize("over,status", [
    (dict(A=None), "DG_ERR_INVALID_ARG"),
    (dict(B=None), "DG_ERR_INVALID_ARG"),
    (dict(C=None), "DG_ERR_INVALID_ARG"),
    (dict(A=0x10008), "DG_ERR_INVALID_ARG"),           # not 16-byte aligned
    (dict(C=0x30002), "DG_ERR_INVALID_ARG"),
    (dict(lda=32), "DG_ERR_INVALID_ARG"),               # lda < K
    (dict(ldb=63, K=60), "DG_ERR_INVALID_ARG"),         # ldb*2 bytes not a multiple of 16
    (dict(M=-1), "DG_ERR_INVALID_ARG"),
    (dict(K=-5), "DG_ERR_INVALID_ARG"),
    (dict(epilogue="bias"), "DG_ERR_INVALID_ARG"),      # bias epilogue, null bias
    (dict(bias=0x40001, epilogue="bias"), "DG_ERR_INVALID_ARG"),
    (dict(dtype_a="i8", dtype_b="f16"), "DG_ERR_UNSUPPORTED"),
    (dict(dtype_a="e2m1", dtype_b="f16"), "DG_ERR_UNSUPPORTED"),
    (dict(dtype_a="i8", dtype_b="i8", epilogue="gelu"), "DG_ERR_UNSUPPORTED"),
    (dict(dtype_a="i8", dtype_b="i8", alpha=1.5), "DG_ERR_UNSUPPORTED"),
    (dict(dtype_a="i8", dtype_b="i8", beta=float("nan")), "DG_ERR_UNSUPPORTED"),
    (dict(dtype_b="e2m1", ldb=63), "DG_ERR_INVALID_ARG"),   # odd E2M1 leading dimension
    (dict(dtype_b="e2m1", ldb=80), "DG_ERR_INVALID_ARG"),   # 40-byte packed rows
    (dict(alpha=float("inf")), "DG_ERR_INVALID_ARG"),
])
def test_invalid_arguments_rejected(dg, over, status):
    got, msg = _call(dg, **over)
    assert got == status, msg
    assert msg  # a message is set


GOOD_EX = dict(M=64, N=64, K=64, dtype_a="f16", dtype_b="f16", A=0x10000, lda=64, B=0x20000,
               ldb=64, C=0x30000, ldc=64, D=0x50000, ldd=72, bias=None, alpha=1.0, beta=1.0,
               program=[])


def _call_ex(dg, **over):
    kw = dict(GOOD_EX)
    kw.update(over)
    prog = kw["program"]
    try:
        dg.gemm_ex_raw(kw["M"], kw["N"], kw["K"], kw["dtype_a"], kw["dtype_b"], kw["A"],
                       kw["lda"], kw["B"], kw["ldb"], kw["C"], kw["ldc"], kw["D"], kw["ldd"],
                       kw["bias"], kw["alpha"], kw["beta"], program=prog, stream=0)
    except dg.DgError as e:
        return e.name, str(e)
    return "DG_OK", ""


def _nine_ops(dg):
    p = dg.make_program(["relu"] * 8)
    p.n_ops = 9
    return p


@pytest.mark.parametrize("over,status", [
    (dict(D=None), "DG_ERR_INVALID_ARG"),
    (dict(D=0x50004), "DG_ERR_INVALID_ARG"),
    (dict(C=None), "DG_ERR_INVALID_ARG"),                  # beta != 0 needs C
    (dict(C=0x30008), "DG_ERR_INVALID_ARG"),
    (dict(ldc=63), "DG_ERR_INVALID_ARG"),                  # ldc < N
    (dict(ldd=32), "DG_ERR_INVALID_ARG"),                  # ldd < N
    (dict(C=0x50000, ldc=64), "DG_ERR_INVALID_ARG"),       # C == D with ldc != ldd
    (dict(program=["bias"]), "DG_ERR_INVALID_ARG"),        # bias op, null bias
    (dict(program=[("clamp", 1.0, -1.0)]), "DG_ERR_INVALID_ARG"),
    (dict(program=[("clamp", float("nan"), 1.0)]), "DG_ERR_INVALID_ARG"),
    (dict(program=[("scale", float("inf"))]), "DG_ERR_INVALID_ARG"),
    (dict(program=[(9, 0.0, 0.0)]), "DG_ERR_INVALID_ARG"),  # unknown op type
    (dict(program=[(0, 0.0, 0.0)]), "DG_ERR_INVALID_ARG"),
    (dict(program="nine"), "DG_ERR_INVALID_ARG"),          # n_ops above the maximum
    (dict(dtype_a="i8", dtype_b="i8", program=["relu"]), "DG_ERR_UNSUPPORTED"),
    (dict(program=[("quant_i8", 1.0), "relu"]), "DG_ERR_INVALID_ARG"),   # quantization not last
    (dict(program=[("quant_i8", float("inf"))]), "DG_ERR_INVALID_ARG"),
    (dict(C=0x50000, ldc=72, program=[("quant_i8", 1.0)]), "DG_ERR_INVALID_ARG"),  # int8 D is C
])
def test_gemm_ex_invalid_arguments_rejected(dg, over, status):
    if over.get("program") == "nine":
        over = dict(over, program=_nine_ops(dg))
    got, msg = _call_ex(dg, **over)
    assert got == status, msg
    assert msg


def test_gemm_ex_unused_c_may_be_null(dg):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # beta == 0: C is not read, so a null C (and any ldc) passes validation and
    # the call reaches the device check
    got, msg = _call_ex(dg, C=None, ldc=0, beta=0.0, program=["relu", ("scale", 2.0)])
    assert got == "DG_ERR_INVALID_STATE", msg


def test_make_program_limits(dg):
    with pytest.raises(ValueError):
        dg.make_program(["relu"] * 9)
    p = dg.make_program(["bias", ("scale", 0.5), ("clamp", -1, 1), "gelu"])
    assert p.n_ops == 4
    assert [p.ops[k].type for k in range(4)] == [1, 4, 5, 3]
    assert (p.ops[1].a, p.ops[2].a, p.ops[2].b) == (0.5, -1.0, 1.0)


def _call_batched(dg, **over):
    kw = dict(batch=4, M=1, N=128, K=4096, dtype_a="f16", dtype_b="f16", A=0x10000, lda=4096,
              sa=4096, B=0x20000, ldb=4096, sb=128 * 4096, C=0x30000, sc=128, bias=None,
              sbias=0, alpha=1.0, beta=0.0, epilogue="none")
    kw.update(over)
    try:
        dg.gemm_strided_batched_raw(kw["batch"], kw["M"], kw["N"], kw["K"], kw["dtype_a"],
                                    kw["dtype_b"], kw["A"], kw["lda"], kw["sa"], kw["B"],
                                    kw["ldb"], kw["sb"], kw["C"], kw["sc"], kw["bias"],
                                    kw["sbias"], kw["alpha"], kw["beta"], kw["epilogue"],
                                    stream=0)
    except dg.DgError as e:
        return e.name, str(e)
    return "DG_OK", ""


@pytest.mark.parametrize("over,status", [
    (dict(batch=-1), "DG_ERR_INVALID_ARG"),
    (dict(sa=-8), "DG_ERR_INVALID_ARG"),
    (dict(sbias=-1), "DG_ERR_INVALID_ARG"),
    (dict(sc=120), "DG_ERR_INVALID_ARG"),            # outputs overlap
    (dict(sa=4100), "DG_ERR_INVALID_ARG"),           # 8200 bytes: not a multiple of 16
    (dict(dtype_b="e2m1", sb=16), "DG_ERR_INVALID_ARG"),   # 8 bytes of codes
    (dict(epilogue="bias"), "DG_ERR_INVALID_ARG"),   # null bias
    (dict(epilogue="sigmoid"), "DG_ERR_INVALID_ARG"),
    (dict(C=None), "DG_ERR_INVALID_ARG"),
])
def test_batched_invalid_arguments_rejected(dg, over, status):
    if over.get("epilogue") == "sigmoid":
        over = dict(over, epilogue=7)
    got, msg = _call_batched(dg, **over)
    assert got == status, msg
    assert msg


def test_batched_empty_is_a_noop(dg):
    assert _call_batched(dg, batch=0, A=None, B=None, C=None)[0] == "DG_OK"
    assert _call_batched(dg, M=0)[0] == "DG_OK"
    # one problem: any stride, as the strides are never applied
    import torch
    if not torch.cuda.is_available():
        assert _call_batched(dg, batch=1, sc=3, sa=1)[0] == "DG_ERR_INVALID_STATE"


def _call_grouped(dg, Ms, A=0x10000, B=0x20000, C=0x30000, bias=None, N=128, K=256,
                  epilogue=0, arrays=True, count=None):
    import ctypes
    n = len(Ms) if count is None else count
    vp = ctypes.c_void_p
    size = max(len(Ms), 1)
    ms = (ctypes.c_int64 * size)(*Ms) if arrays else None
    pa = (vp * size)(*[A] * len(Ms)) if arrays else None
    pb = (vp * size)(*[B] * len(Ms)) if arrays else None
    pc = (vp * size)(*[C] * len(Ms)) if arrays else None
    pbias = None if bias is None else (vp * size)(*[bias] * len(Ms))
    st = dg.lib().dg_gemm_grouped(n, ms, N, K, 0, 0, pa, 256, pb, 256, pc, pbias, 1.0, 0.0,
                                  epilogue, None)
    return st, dg.last_error()


def test_grouped_invalid_arguments_rejected(dg):
    assert _call_grouped(dg, [1, 2], count=-1)[0] == 1
    assert _call_grouped(dg, [1, 2], arrays=False)[0] == 1
    st, msg = _call_grouped(dg, [1, -3])
    assert st == 1 and "negative M" in msg
    st, msg = _call_grouped(dg, [1, 2], epilogue=1)     # bias epilogue, no bias array
    assert st == 1 and "bias" in msg
    st, msg = _call_grouped(dg, [4, 2], A=0x10008)      # misaligned A, reported per problem
    assert st == 1 and msg.startswith("problem 0:")
    assert _call_grouped(dg, [], count=0)[0] == 0
    assert _call_grouped(dg, [0, 0])[0] == 0            # nothing to do


def test_empty_problem_is_a_noop(dg):
    assert _call(dg, M=0)[0] == "DG_OK"
    assert _call(dg, N=0, A=None, B=None)[0] == "DG_OK"


def test_valid_call_without_gpu_reports_state(dg):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    got, msg = _call(dg)
    assert got == "DG_ERR_INVALID_STATE", msg


def test_last_error_is_cleared_by_next_call(dg):
    _call(dg, A=None)
    assert dg.last_error()
    dg.set_wait_timeout_ns(0)
    assert dg.last_error() == ""


def test_launch_count_readable(dg):
    assert dg.launch_count() >= 0


def test_product_does_not_import_oracle():
    pkg = os.path.join(ROOT, "precision_matmul_dg_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.replace("oracle-free", ""), f


# ---------------------------------------------------------------- MXFP4 entry points

QGOOD = dict(rows=64, K=64, X=0x10000, ldx=64, codes=0x20000, ldq=64, scales=0x30000, lds=2)


@pytest.mark.parametrize("over", [
    dict(rows=-1), dict(K=-3), dict(X=None), dict(X=0x10008), dict(ldx=68), dict(ldx=32),
    dict(codes=None), dict(codes=0x20004), dict(ldq=80), dict(ldq=32), dict(scales=None),
    dict(lds=1),
], ids=lambda o: ",".join("%s=%s" % kv for kv in o.items()))
def test_quantize_mxf4_invalid_arguments_rejected(dg, over):
    kw = dict(QGOOD)
    kw.update(over)
    with pytest.raises(dg.DgError) as ei:
        dg.quantize_mxf4_raw(stream=0, **kw)
    assert ei.value.name == "DG_ERR_INVALID_ARG"


def test_quantize_mxf4_empty_is_a_noop(dg):
    dg.quantize_mxf4_raw(0, 64, None, 64, None, 64, None, 2, stream=0)
    dg.quantize_mxf4_raw(64, 0, None, 64, None, 64, None, 2, stream=0)


MGOOD = dict(M=64, N=64, K=64, A=0x10000, lda=64, scale_a=0x11000, lds_a=2, B=0x20000, ldb=64,
             scale_b=0x21000, lds_b=2, C=0x30000, bias=None, alpha=1.0, beta=0.0,
             epilogue="none")


@pytest.mark.parametrize("over", [
    dict(M=-1), dict(A=None), dict(scale_a=None), dict(B=None), dict(scale_b=None),
    dict(C=None), dict(C=0x30002), dict(A=0x10008), dict(lda=80), dict(lda=32), dict(ldb=104),
    dict(lds_a=1), dict(lds_b=1), dict(epilogue="bias"), dict(alpha=float("nan")),
    dict(bias=0x40001, epilogue="bias_gelu"),
], ids=lambda o: ",".join("%s=%s" % kv for kv in o.items()))
def test_gemm_mxf4_invalid_arguments_rejected(dg, over):
    kw = dict(MGOOD)
    kw.update(over)
    with pytest.raises(dg.DgError) as ei:
        dg.gemm_mxf4_raw(stream=0, **kw)
    assert ei.value.name == "DG_ERR_INVALID_ARG"


def test_gemm_mxf4_empty_is_a_noop(dg):
    for M, N in ((0, 64), (64, 0)):
        dg.gemm_mxf4_raw(M, N, 64, None, 64, None, 2, None, 64, None, 2, None, None, 1.0, 0.0,
                         stream=0)


def test_mxf4_pair_is_for_its_own_entry_point(dg):
    # dg_gemm and dg_gemm_ex take no scales: the MXF4 pair is refused there
    for pair in (("mxf4", "mxf4"), ("f16", "mxf4"), ("mxf4", "f16")):
        got, _ = _call(dg, dtype_a=pair[0], dtype_b=pair[1])
        assert got == "DG_ERR_UNSUPPORTED", pair
