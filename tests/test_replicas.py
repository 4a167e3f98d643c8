"""The N > 1 host logic of bench.py on CPU (gloo, world size 2): the path is
replicas only (no collective on the data path), so what runs across ranks is
the rendezvous, the barriers and the max / sum over ranks of the timings."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    mx = bench.max_over_ranks(1.5 + rank, w)
    sm = bench.sum_over_ranks(10.0 * (rank + 1), w)
    out.put((rank, mx, sm, dist.get_backend()))
    bench.barrier(w)
    dist.destroy_process_group()


def test_max_and_sum_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    # every rank sees the maximum time (slowest rank) and the total work
    assert [g[1] for g in got] == [2.5, 2.5]
    assert [g[2] for g in got] == [30.0, 30.0]
    assert {g[3] for g in got} == {"gloo"}


def test_reference_arm_under_torchrun_prints_one_line():
    # rank 0 alone runs the oracle arm and prints one JSON line; rank 1 exits 0
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
           "thin_1x256x12800", "--steps", "2", "--warmup", "3", "--gpus", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
