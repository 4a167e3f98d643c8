"""The planner's register constraint on a GB300: it is checked against the
registers ptxas actually gave each kernel (read with cudaFuncGetAttributes),
not against a fixed bound (kwkr.cn/news/562171, section 2.2 first layer:
register use no larger than the registers available)."""

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    import __graft_entry__
    __graft_entry__.build()
    import precision_matmul_dg_gb300 as dg
    assert torch.cuda.is_available()
    return dg


def _variants(plans, kernel):
    return {(p["n_tile"], p["stages"], p["cta_group"]): p for p in plans
            if p["kernel_name"] == kernel}


@pytest.mark.parametrize("shape,dtypes,kernel", [
    ((4096, 4096, 4096), ("f16", "f16"), "tc"),
    ((4096, 4096, 4096), ("i8", "i8"), "tc_widened"),
    ((1, 4096, 65536), ("f16", "f16"), "gemv"),
    ((8, 4096, 65536), ("f16", "f16"), "gemv_mma"),
    ((16, 8960, 1536), ("f16", "e2m1"), "skinny")])
def test_register_constraint_uses_measured_figures(dg, shape, dtypes, kernel):
    M, N, K = shape
    hw = dg.query_hw().as_dict()
    plans = _variants(dg.plan_tiles(M, N, K, *dtypes, hw=hw), kernel)
    assert plans, kernel
    key, p = sorted(plans.items())[0]
    regs = p["regs_per_thread"]
    assert 0 < regs <= 255
    # a descriptor with exactly the registers that variant's CTA needs keeps
    # it; one register fewer per SM prunes it
    enough = dict(hw, regs_per_sm=regs * p["threads"])
    short = dict(hw, regs_per_sm=regs * p["threads"] - 1)
    assert key in _variants(dg.plan_tiles(M, N, K, *dtypes, hw=enough), kernel)
    try:
        left = _variants(dg.plan_tiles(M, N, K, *dtypes, hw=short), kernel)
    except dg.DgError as e:   # nothing left at all
        assert e.name == "DG_ERR_NO_VALID_CANDIDATE"
        left = {}
    assert key not in left
