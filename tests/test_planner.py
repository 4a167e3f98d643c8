"""Planner properties (host only).

The constraint system (kwkr.cn "DeepGEMM" article, section 2.2 first layer):
shared memory <= available, registers <= available, occupancy >= target.
Each returned plan is re-checked here against those constraints written out
independently, and the returned set is compared with a brute-force
enumeration of the compiled tile space.
"""

import math
import os

import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# A GB300-like description (152 SMs, 227 KB per CTA, 512 TMEM columns).
GB300 = dict(sm_count=152, cc_major=10, cc_minor=3, smem_per_block_optin=232448,
             smem_per_sm=233472, regs_per_sm=65536, regs_per_thread_max=255,
             max_threads_per_sm=2048, tmem_cols=512, l2_bytes=126 * 1024 * 1024,
             hbm_gbps=6800.0, tc_f16_tflops=1900.0, clock_ghz=2.07)

# Compiled FP16 tensor-core variants: (N_tile, stages, CTAs per tile); M_tile
# 128 per CTA, K_tile 64, 384 threads.  A CTA pair holds half of B per CTA.
TC_VARIANTS = [(256, 4, 1), (128, 6, 1), (64, 8, 1), (256, 6, 2), (224, 6, 2), (192, 6, 2),
               (128, 8, 2)]
# The output passes through two 2 KB staging boxes per epilogue warp (8 warps)
EPI_STAGING = 8 * 2 * 32 * 32 * 2


@pytest.fixture(scope="module")
def dg():
    import __graft_entry__
    __graft_entry__.build()
    import precision_matmul_dg_gb300 as dg
    return dg


def tc_smem(n_tile, stages, cg=1, staged=True):
    return (stages * (128 * 64 * 2 + (n_tile // cg) * 64 * 2) + (EPI_STAGING if staged else 0)
            + 512 + 1024)


def tc_feasible(M, N, hw, target):
    out = set()
    for n_tile, stages, cg in TC_VARIANTS:
        if cg == 2 and M <= 128:      # a pair needs more than one CTA's rows
            continue
        if tc_smem(n_tile, stages, cg) > hw["smem_per_block_optin"]:
            continue
        if 2 * n_tile > hw["tmem_cols"]:
            continue
        if 384 * 168 > hw["regs_per_sm"]:
            continue
        units = hw["sm_count"] // cg
        tiles = math.ceil(M / (128 * cg)) * math.ceil(N / n_tile)
        waves = math.ceil(tiles / units)
        if tiles / (waves * units) < target:
            continue
        out.add(("tc", n_tile, stages, cg))
    return out


# FP16 tensor-core variants also compiled with stream-K work division
SK_VARIANTS = [(256, 6, 2), (128, 6, 1)]


def stream_k_model(tiles, kb, units):
    """The stream-K division as the kernel documents it, by brute force.
    Fewer tiles than units: every tile cut into p = units // tiles equal
    ranges (at most 4, each at least 4 K blocks; none when p < 2).  Else
    whole tiles for all but the last ragged wave and the wave before it, the
    K blocks of those tiles dealt out in even contiguous ranges (at least half
    a tile and 4 K blocks each).  The pieces of each tile are counted by
    scanning its K blocks.  Returns (dp_tiles, sk_units, max_pieces, longest
    range) or None when there is nothing to balance."""
    if kb < 2 or units < 2 or tiles % units == 0:
        return None
    if tiles < units:
        p = min(units // tiles, 4, kb // 4)
        if p < 2:
            return None
        sk_tiles, n = tiles, tiles * p
    else:
        sk_tiles = tiles % units + units
        n = min(units, 2 * sk_tiles, max(1, sk_tiles * kb // 4))
    iters = sk_tiles * kb
    bounds = [u * iters // n for u in range(n + 1)]
    owner = []
    for u in range(n):
        owner += [u] * (bounds[u + 1] - bounds[u])
    assert len(owner) == iters and all(bounds[u + 1] > bounds[u] for u in range(n))
    pieces = max(len(set(owner[t * kb:(t + 1) * kb])) for t in range(sk_tiles))
    longest = max(bounds[u + 1] - bounds[u] for u in range(n))
    return tiles - sk_tiles, n, pieces, longest


def sk_feasible(M, N, K, hw, target):
    out = {}
    kb = math.ceil(K / 64)
    for n_tile, stages, cg in SK_VARIANTS:
        if cg == 2 and M <= 128:
            continue
        if tc_smem(n_tile, stages, cg) > hw["smem_per_block_optin"] or 2 * n_tile > hw["tmem_cols"]:
            continue
        if 384 * 168 > hw["regs_per_sm"]:
            continue
        units = hw["sm_count"] // cg
        tiles = math.ceil(M / (128 * cg)) * math.ceil(N / n_tile)
        if tiles >= units:            # proposed only below one wave of tiles
            continue
        m = stream_k_model(tiles, kb, units)
        if m is None:
            continue
        dp, n, pieces, longest = m
        occ = tiles * kb / (units * (dp // units * kb + longest))
        if occ >= target:
            out[("tc_streamk", n_tile, stages, cg)] = (pieces, cg * units)
    return out


def gemv_feasible(M, N, K, hw, target):
    out = set()
    if M > 8:
        return out
    resident = hw["sm_count"] * 64
    for split in GEMV_SPLITS:
        chunk = math.ceil(math.ceil(K / split) / 256) * 256
        if split > 1 and chunk * (split - 1) >= K:
            continue                      # the last split would be empty
        units = N * split
        waves = math.ceil(units / resident)
        if units / (waves * resident) >= target:
            out.add(("gemv", 8, 1, split))
    return out


GEMV_SPLITS = [1, 2, 3, 4, 5, 6, 7, 8, 10, 12, 13, 14, 16, 20, 24, 28, 32, 40, 48, 64, 96, 128,
               160, 192, 256]


def gemv_mma_feasible(M, N, K, hw, target):
    # warp-MMA GEMV: 2 <= M <= 16; CTAs of 256 threads at 80 registers, a
    # warp per 8 columns
    out = set()
    if not 2 <= M <= 16:
        return out
    ctas = hw["regs_per_sm"] // (80 * 256)
    resident = hw["sm_count"] * ctas * 8
    for split in GEMV_SPLITS:
        chunk = math.ceil(math.ceil(K / split) / 256) * 256
        if split > 1 and chunk * (split - 1) >= K:
            continue
        units = math.ceil(N / 8) * split
        waves = math.ceil(units / resident)
        if units / (waves * resident) >= target:
            out.add(("gemv_mma", 64, 1, split))
    return out


SHAPES = [(256, 256, 256), (4096, 4096, 4096), (2048, 2048, 2048), (8192, 8192, 8192),
          (1, 4096, 131072), (1, 256, 12800), (7, 1000, 999), (300, 520, 200), (129, 17, 64)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("target", [0.0, 0.5, 0.7, 0.9])
def test_plans_satisfy_constraints_and_match_enumeration(dg, shape, target):
    M, N, K = shape
    sk = sk_feasible(M, N, K, GB300, target)
    want = (tc_feasible(M, N, GB300, target) | gemv_feasible(M, N, K, GB300, target) |
            gemv_mma_feasible(M, N, K, GB300, target) | set(sk))
    if not want:
        with pytest.raises(dg.DgError) as ei:
            dg.plan_tiles(M, N, K, hw=GB300, target_occupancy=target)
        assert ei.value.name == "DG_ERR_NO_VALID_CANDIDATE"
        assert "no valid candidate" in str(ei.value)
        return
    plans = dg.plan_tiles(M, N, K, hw=GB300, target_occupancy=target)
    got = set()
    for p in plans:
        assert p["occupancy"] >= target - 1e-12
        if p["kernel_name"] == "tc":
            cg = p["cta_group"]
            assert p["smem_bytes"] == tc_smem(p["n_tile"], p["stages"], cg)
            assert p["smem_bytes"] <= GB300["smem_per_block_optin"]
            assert 2 * p["n_tile"] <= GB300["tmem_cols"]
            # the kernel's measured registers with a device, else the bound 168
            assert 0 < p["regs_per_thread"] <= 168
            assert p["threads"] * p["regs_per_thread"] <= GB300["regs_per_sm"]
            tiles = math.ceil(M / (128 * cg)) * math.ceil(N / p["n_tile"])
            assert p["grid"] == cg * min(tiles, GB300["sm_count"] // cg)
            assert p["m_tile"] == 128 * cg and p["k_tile"] == 64 and p["split_k"] == 1
            got.add(("tc", p["n_tile"], p["stages"], cg))
        elif p["kernel_name"] == "tc_streamk":
            cg = p["cta_group"]
            key = ("tc_streamk", p["n_tile"], p["stages"], cg)
            assert key in sk
            assert p["smem_bytes"] == tc_smem(p["n_tile"], p["stages"], cg)
            assert 0 < p["regs_per_thread"] <= 168
            assert p["m_tile"] == 128 * cg and p["k_tile"] == 64
            # split_k: the most ranges one tile is cut into; grid: the CTAs
            # the work is divided over
            assert (p["split_k"], p["grid"]) == sk[key]
            got.add(key)
        else:
            assert p["kernel_name"] in ("gemv", "gemv_mma")
            assert p["k_tile"] % 256 == 0
            assert p["k_tile"] * p["split_k"] >= K
            assert p["k_tile"] * (p["split_k"] - 1) < K      # no empty split
            got.add((p["kernel_name"], p["n_tile"], p["stages"], p["split_k"]))
    assert got == want
    # ranked by estimated time
    ests = [p["est_us"] for p in plans]
    assert ests == sorted(ests)


def test_stream_k_division():
    # 2048^3 in 256 x 256 pair tiles: 64 tiles on 76 pairs, no two pairs per
    # tile: nothing to balance
    assert stream_k_model(64, 32, 76) is None
    # 16 tiles of 256 K blocks on 76 pairs: four equal pieces per tile
    assert stream_k_model(16, 256, 76) == (0, 64, 4, 64)
    # 4096^3: 256 tiles, 3 whole waves and 28 left: 2 waves stay whole
    dp, n, pieces, longest = stream_k_model(256, 64, 76)
    assert (dp, n, pieces) == (152, 76, 2) and longest == 88
    # one tile of 8 K blocks: two ranges of 4
    assert stream_k_model(1, 8, 76) == (0, 2, 2, 4)
    # 64 tiles of 256 K blocks on 152 CTAs: two halves per tile
    assert stream_k_model(64, 256, 152) == (0, 128, 2, 128)
    # one tile of 9 K blocks: two ranges (of at least 4)
    assert stream_k_model(1, 9, 76) == (0, 2, 2, 5)
    # whole waves, or a single K block: nothing to balance
    assert stream_k_model(152, 64, 76) is None and stream_k_model(10, 1, 76) is None


def test_stream_k_plans_below_one_wave(dg):
    # 256 x 4096 x 16384: 16 pair tiles of 256 x 256 on 76 pairs, 64 tiles of
    # 128 x 128 on 152 CTAs: both divided by K, and ranked first
    plans = dg.plan_tiles(256, 4096, 16384, hw=GB300, target_occupancy=0.0)
    sk = [p for p in plans if p["kernel_name"] == "tc_streamk"]
    assert {(p["n_tile"], p["cta_group"]) for p in sk} == {(256, 2), (128, 1)}
    assert plans[0]["kernel_name"] == "tc_streamk"
    # more tiles than units (2560^2 x 4096: 100 pair tiles, 400 single tiles):
    # whole waves, no stream-K plan
    plans = dg.plan_tiles(2560, 2560, 4096, hw=GB300, target_occupancy=0.0)
    assert not [p for p in plans if p["kernel_name"] == "tc_streamk"]
    # other dtype pairs have none
    assert not [p for p in dg.plan_tiles(256, 4096, 16384, "i8", "i8", hw=GB300)
                if p["kernel_name"] == "tc_streamk"]


def test_resources_prune(dg):
    tiny = dict(GB300, smem_per_block_optin=64 * 1024)
    with pytest.raises(dg.DgError) as ei:
        dg.plan_tiles(4096, 4096, 4096, hw=tiny)
    assert ei.value.name == "DG_ERR_NO_VALID_CANDIDATE"
    # every compiled variant needs tc_smem(...) bytes; one byte less prunes it
    for n, s, cg in TC_VARIANTS:
        tight = dict(GB300, smem_per_block_optin=tc_smem(n, s, cg) - 1)
        try:
            plans = dg.plan_tiles(4096, 4096, 4096, hw=tight)
        except dg.DgError:
            plans = []
        assert (n, s, cg) not in {(p["n_tile"], p["stages"], p["cta_group"]) for p in plans}
    small_tmem = dict(GB300, tmem_cols=256)
    assert {p["n_tile"] for p in dg.plan_tiles(4096, 4096, 4096, hw=small_tmem)} == {64, 128}


def test_dtype_pairs(dg):
    with pytest.raises(dg.DgError) as ei:
        dg.plan_tiles(64, 64, 64, "i8", "f16", hw=GB300)
    assert ei.value.name == "DG_ERR_UNSUPPORTED"


def test_bad_planner_arguments(dg):
    for bad in [dict(M=0), dict(K=-1), dict(target_occupancy=1.5)]:
        kw = dict(M=64, N=64, K=64, hw=GB300, target_occupancy=0.0)
        kw.update(bad)
        with pytest.raises(dg.DgError) as ei:
            dg.plan_tiles(kw["M"], kw["N"], kw["K"], hw=kw["hw"],
                          target_occupancy=kw["target_occupancy"])
        assert ei.value.name == "DG_ERR_INVALID_ARG"


def _golden_a100():
    d, tiles = {}, []
    for line in open(os.path.join(GOLDEN, "planner_a100_example.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, *v = line.split()
        if k == "tile":
            tiles.append(tuple(int(x) for x in v))
        else:
            d[k] = v
    return d, tiles


def test_worked_example_tiles_fit_the_a100_description(dg):
    """The article's A100 example: its three printed tiles satisfy the shared
    memory constraint of the printed hardware description and are among the
    planner's warp-MMA candidates.  The printed GFLOPS estimates and the count
    of 7 solutions rest on a cost model the article does not give and are not
    reproduced (parity unpinned)."""
    d, tiles = _golden_a100()
    smem = int(d["shared_memory_per_sm_kb"][0]) * 1024
    cc = d["compute_capability"][0].split(".")
    hw = dict(sm_count=108, cc_major=int(cc[0]), cc_minor=int(cc[1]), smem_per_block_optin=smem,
              smem_per_sm=smem, regs_per_sm=65536, regs_per_thread_max=255,
              max_threads_per_sm=int(d["max_threads_per_sm"][0]), tmem_cols=0,
              l2_bytes=int(d["l2_cache_size_kb"][0]) * 1024, hbm_gbps=1555.0,
              tc_f16_tflops=312.0, clock_ghz=1.41)
    M, N, K = (int(x) for x in d["shape"])
    plans = dg.plan_tiles(M, N, K, hw=hw, target_occupancy=0.0, max_out=4096)
    got = {(p["m_tile"], p["n_tile"], p["k_tile"]) for p in plans}
    for t in tiles:
        assert t in got, t
        assert 2 * (t[0] + t[1]) * t[2] * 2 <= smem
    assert all(p["kernel_name"] == "none" for p in plans)  # planning only: no kernel here


# converting kernel: (N_tile, input-ring slots) and the widened-operand slots
CONV_VARIANTS = {("i8", "i8"): [(128, 8)], ("f16", "e2m1"): [(256, 6), (128, 8), (64, 8)]}
CV_SLOTS = {("i8", "i8", 128): 3, ("f16", "e2m1", 256): 2, ("f16", "e2m1", 128): 3,
            ("f16", "e2m1", 64): 4}


def conv_smem(da, db, n_tile, stages):
    in_a = 128 * 64 if da == "i8" else 128 * 64 * 2
    in_b = n_tile * 64 if db == "i8" else n_tile * 32
    cv = (128 * 64 * 2 if da == "i8" else 0) + n_tile * 64 * 2
    return stages * (in_a + in_b) + CV_SLOTS[(da, db, n_tile)] * cv + 512 + 1024


@pytest.mark.parametrize("pair", sorted(CONV_VARIANTS))
@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (16, 8960, 1536), (2048, 8960, 1536),
                                   (7, 9, 5)])
def test_converting_kernel_plans(dg, pair, shape):
    M, N, K = shape
    plans = dg.plan_tiles(M, N, K, pair[0], pair[1], hw=GB300, target_occupancy=0.0)
    skinny = pair == ("f16", "e2m1") and M <= 16
    assert {p["kernel_name"] for p in plans} == {"tc", "tc_widened"} | ({"skinny"} if skinny else set())
    conv = [p for p in plans if p["kernel_name"] == "tc" and not p["swap_ab"]]
    assert {(p["n_tile"], p["stages"]) for p in conv} == set(CONV_VARIANTS[pair])
    # FP16 x E2M1 also: the weights widened in tensor memory, D^T tiles of 128
    # weight rows x 160 or 224 activation rows (7 or 6 stages of an activation
    # tile and 4 KB of codes, 32 KB of epilogue boxes), 448 threads
    swapped = [p for p in plans if p["kernel_name"] == "tc" and p["swap_ab"]]
    if pair == ("f16", "e2m1"):
        assert sorted((p["m_tile"], p["n_tile"], p["stages"], p["cta_group"]) for p in swapped) == \
            [(128, 160, 7, 1), (128, 224, 6, 1)]
        for w4t in swapped:
            bn, st = w4t["n_tile"], w4t["stages"]
            assert w4t["threads"] == 448
            assert w4t["smem_bytes"] == st * (bn * 128 + 128 * 32) + 8 * 2 * 2048 + 1024 + 512
            assert w4t["smem_bytes"] <= GB300["smem_per_block_optin"]
            assert w4t["grid"] == min(152, math.ceil(N / 128) * math.ceil(M / bn))
    else:
        assert not swapped
    for p in conv:
        assert p["threads"] == 384
        assert p["smem_bytes"] == conv_smem(pair[0], pair[1], p["n_tile"], p["stages"])
        assert p["smem_bytes"] <= GB300["smem_per_block_optin"]
        cols = (3 if pair[0] == "i8" else 2) * p["n_tile"]
        assert cols <= GB300["tmem_cols"]
    # widened: the FP16 kernel's variants (INT8: its exact-INT32 mode, 128 x 128,
    # 256 x 192 and 256 x 224)
    wide = {(p["n_tile"], p["stages"], p["cta_group"]) for p in plans
            if p["kernel_name"] == "tc_widened"}
    if pair[0] == "i8":
        want = {(128, 6, 1), (192, 6, 2), (224, 6, 2)}
    else:
        want = set(TC_VARIANTS)
    if M <= 128:
        want = {w for w in want if w[2] == 1}
    assert wide == want
    for p in plans:
        if p["kernel_name"] == "tc_widened":
            assert p["threads"] == 384
            # INT8 runs the FP16 kernel in its exact INT32 mode (also staged)
            assert p["smem_bytes"] == tc_smem(p["n_tile"], p["stages"], p["cta_group"])


@pytest.mark.parametrize("M", [1, 7, 16, 17])
def test_skinny_plans(dg, M):
    # FP16 x E2M1 with M <= 16: one 512-thread block per 64 columns, 2048-code
    # activation chunks in shared memory split between two warp halves
    N, K = 8960, 1536
    plans = dg.plan_tiles(M, N, K, "f16", "e2m1", hw=GB300, target_occupancy=0.0)
    sk = [p for p in plans if p["kernel_name"] == "skinny"]
    if M > 16:
        assert not sk
        return
    assert len(sk) == 1
    p = sk[0]
    assert (p["m_tile"], p["n_tile"], p["k_tile"], p["split_k"]) == (16, 64, 2048, 2)
    assert p["threads"] == 512 and p["grid"] == math.ceil(N / 64)
    assert p["smem_bytes"] == 16 * 2048 * 2 + 16 * (2048 + 8) * 2 + 8 * 32 * 4 * 4
    assert p["smem_bytes"] <= GB300["smem_per_block_optin"]
    # it streams the weights once: ranked first for the HBM-bound shape
    assert plans[0]["kernel_name"] == "skinny"
    # not for other dtype pairs
    assert not [q for q in dg.plan_tiles(M, N, K, "f16", "f16", hw=GB300, target_occupancy=0.0)
                if q["kernel_name"] == "skinny"]


def mx_smem(n_tile, stages, cg):
    # 128-byte rows of packed codes for A (128 rows) and B (a CTA of a pair
    # holds half of the tile's rows), the stage's scale images (1 KB per 128
    # rows: this CTA's A rows and the whole B tile) and the 16 row-major
    # scale bytes per row they are built from (128 rows of A, n_tile of B),
    # the FP16 output staging boxes, barriers and the 1 KB alignment slack
    return (stages * (128 * 128 + (n_tile // cg) * 128 + 1024 * (1 + math.ceil(n_tile / 128))
                      + 16 * (128 + n_tile))
            + EPI_STAGING + 512 + 1024)


def test_mxf4_plans(dg):
    # MXFP4 runs on the block-scaled MMA (kernel "tc", 256 values of K per
    # stage) or through the BF16 widening ("tc_widened"); every native plan
    # fits the shared memory and tensor memory (two accumulators plus two
    # buffers of scale words), and an odd K leaves only the widening
    for shape in [(1, 4096, 4096), (16, 8960, 1536), (4096, 4096, 4096), (130, 1000, 1000)]:
        plans = dg.plan_tiles(*shape, "mxf4", "mxf4", hw=GB300, max_out=64)
        assert {p["kernel_name"] for p in plans} == {"tc", "tc_widened"}, shape
        for p in plans:
            if p["kernel_name"] != "tc":
                continue
            cg = p["cta_group"]
            assert (p["m_tile"], p["k_tile"]) == (128 * cg, 256)
            assert (p["n_tile"], p["stages"], cg) in ((224, 3, 1), (128, 5, 1), (224, 5, 2),
                                                      (192, 5, 2))
            assert cg == 1 or shape[0] > 128   # a pair needs more than one CTA's rows
            assert p["smem_bytes"] == mx_smem(p["n_tile"], p["stages"], cg)
            assert p["smem_bytes"] <= GB300["smem_per_block_optin"]
            sf_cols = 2 * (8 + 8 * math.ceil(p["n_tile"] / 128))
            assert 2 * p["n_tile"] + sf_cols <= GB300["tmem_cols"]
    for K in (33, 1001):
        plans = dg.plan_tiles(256, 512, K, "mxf4", "mxf4", hw=GB300, max_out=64)
        assert {p["kernel_name"] for p in plans} == {"tc_widened"}, K
    for pair in (("f16", "mxf4"), ("mxf4", "e2m1")):
        with pytest.raises(dg.DgError) as ei:
            dg.plan_tiles(64, 64, 64, *pair, hw=GB300)
        assert ei.value.name == "DG_ERR_UNSUPPORTED"


def test_noalloc_scratch_covers_every_gemv_split(dg):
    # dg_gemm_thin_noalloc keeps its split-K partials (split * M * N * 4 bytes)
    # and counters (ceil(N / 8) * 4 bytes) in a static array of 2 MiB + 64 KiB
    # and rejects shapes beyond it.  The GEMV's best split (its fastest
    # candidate) stays far below both limits over thin shapes from tiny to huge.
    worst = 0.0
    for M in (1, 2, 4, 8):
        for N in (8, 64, 256, 1024, 4096, 16384, 65536, 131072, 262144):
            for K in (256, 4096, 65536, 1048576, 4194304):
                cands = [p for p in dg.plan_tiles(M, N, K, hw=GB300, target_occupancy=0.0)
                         if p["kernel"] == 1]  # DG_KERNEL_GEMV
                best = min(cands, key=lambda p: p["est_us"])
                if best["split_k"] > 1:
                    worst = max(worst, best["split_k"] * M * N * 4 / (2 << 20))
                    assert (N + 7) // 8 * 4 <= 64 << 10
    assert worst <= 0.25


@pytest.mark.parametrize("n", [4096, 8192])
def test_int8_square_takes_the_224_wide_pair(dg, n):
    # INT8 squares: 256 x 224 pair tiles fill whole waves of 76 pairs at 4096
    # (304 tiles; 256 x 192: 352 tiles, 4.63 waves), and the planner ranks
    # them first; 128 x 128 single CTAs and 256 x 192 pairs stay proposed
    plans = [p for p in dg.plan_tiles(n, n, n, "i8", "i8", hw=GB300)
             if p["kernel_name"] == "tc_widened"]
    assert (plans[0]["n_tile"], plans[0]["stages"], plans[0]["cta_group"]) == (224, 6, 2)
    assert {(p["n_tile"], p["cta_group"]) for p in plans} >= {(128, 1), (192, 2), (224, 2)}
    first = plans[0]
    tiles = math.ceil(n / 256) * math.ceil(n / 224)
    assert first["occupancy"] == pytest.approx(tiles / (math.ceil(tiles / 76) * 76))
