"""Host-side checks of bench.py's workload plumbing (no GPU): every named
workload has a description and a bound, its algorithmic bytes match the
figures worked out by hand for the grouped and MXFP4 cases, and the oracle
rows the CPU legs time are the oracle's own definition."""

import numpy as np
import pytest

import bench
import oracle
import workloads


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_every_workload_is_described(name):
    desc, bound = bench.workload_info(name)
    assert desc and bound in ("tensor", "hbm")


def test_algorithmic_bytes_by_hand():
    # grouped: every expert's weights once, plus each expert's own rows of A and D
    case = workloads.grouped_experts(4, 64, 128, m_hi=4, seed=1)
    rows = sum(case.group_ms)
    assert bench.algorithmic_bytes(case) == 4 * 64 * 128 * 2 + rows * (128 * 2 + 64 * 2)
    assert case.flops() == 2.0 * rows * 64 * 128
    # MXFP4 with FP16 activations: 2 bytes per activation, 0.5 + 1/32 per
    # weight, C read and D written in FP16
    case = workloads.mxf4_case(64, 96, 128, beta=0.5, fp16_a=True)
    want = 64 * 128 * 2 + 96 * 128 * (0.5 + 1 / 32) + 2 * 64 * 96 * 2
    assert bench.algorithmic_bytes(case) == int(want)


def test_oracle_rows_of_the_mxf4_step():
    # the CPU legs of the MXFP4 workload quantize the sampled activation rows
    # and multiply them: the same as quantizing everything, then sampling
    case = workloads.mxf4_case(40, 24, 70, beta=0.5, fp16_a=True, seed=2)
    rows = np.array([0, 7, 39])
    got = bench.oracle_rows(oracle, case, rows)
    codes, scales = oracle.mxfp4_quantize(case.a_fp16, case.K)
    full = oracle.gemm_mx_reference(oracle.pack_e2m1(codes), scales, case.B, case.scale_b,
                                    case.K, C=case.C, alpha=case.alpha, beta=case.beta)
    np.testing.assert_array_equal(got, full[rows])


def test_default_configs_cover_every_measured_configuration():
    # the default line measures the headline plus every configuration of the
    # GEMM (square FP16 at four sizes, INT8, both thin shapes, W4A16 at both
    # M, MXFP4), each once
    class A:
        configs = "default"
    names = bench.config_names(A, "f16_4096")
    assert sorted(names + ["f16_4096"]) == sorted(
        ["f16_256", "f16_2048", "f16_4096", "f16_8192", "i8_4096", "thin_1x4096x131072",
         "thin_1x256x12800", "w4a16_m16", "w4a16_m2048", "mxf4_4096"])
    A.configs = "none"
    assert bench.config_names(A, "f16_4096") == []
    A.configs = "thin_1x256x12800,f16_4096"
    assert bench.config_names(A, "f16_4096") == ["thin_1x256x12800"]
    A.configs = "nonesuch"
    with pytest.raises(SystemExit):
        bench.config_names(A, "f16_4096")
