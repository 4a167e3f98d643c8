"""Several host threads making their first libdg calls at the same moment,
each on its own stream, in a fresh process (so that every kernel's one-time
set-up is still to be done): every result must meet the oracle.  The calls
cover each kernel family the planner picks, so that the threads race on the
set-up of different kernels and on the same one."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (dtype_a, dtype_b, M, N, K): TC single CTA, TC pair, GEMV, warp-MMA GEMV,
# skinny W4A16, TC with in-kernel widening, widened then TC pair, INT8
SHAPES = [("f16", "f16", 512, 1040, 520), ("f16", "f16", 1536, 2000, 512),
          ("f16", "f16", 1, 4000, 3000), ("f16", "f16", 5, 1000, 3000),
          ("f16", "e2m1", 8, 1000, 2048), ("f16", "e2m1", 130, 1000, 512),
          ("f16", "e2m1", 1024, 2048, 1024), ("i8", "i8", 256, 520, 640)]
THREADS_PER_SHAPE = 2
REPEATS = 3


def _child():
    import threading

    import torch

    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import precision_matmul_dg_gb300 as dg
    import workloads
    from gpu_util import assert_parity, to_device

    torch.cuda.init()
    jobs = []
    for i, (da, db, M, N, K) in enumerate(SHAPES * THREADS_PER_SHAPE):
        f16 = da == "f16"  # the INT8 path takes integral alpha and beta only
        case = workloads.random_case(M, N, K, dtype_a=da, dtype_b=db, alpha=0.75 if f16 else 3.0,
                                     beta=0.5 if f16 else 2.0, seed=100 + i,
                                     epilogue="bias_gelu" if f16 else "none")
        jobs.append(case)
    operands = [to_device(c) for c in jobs]
    originals = [o[2].clone() for o in operands]
    torch.cuda.synchronize()
    start = threading.Barrier(len(jobs))
    errors = []
    outs = [None] * len(jobs)

    def work(i):
        try:
            case = jobs[i]
            A, B, C, bias, _ = operands[i]
            stream = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(stream):
                for _ in range(REPEATS):
                    C.copy_(originals[i])
                    dg.gemm(A, B, C, K=case.K, bias=bias, alpha=case.alpha, beta=case.beta,
                            epilogue=case.epilogue, dtype_b=case.dtype_b, stream=stream)
                dg.check_status(stream)
                outs[i] = C.cpu().numpy()
        except Exception as e:  # reported by the main thread
            errors.append("%s: %r" % (jobs[i].name, e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(300)
    assert not any(t.is_alive() for t in threads), "a thread did not finish"
    assert not errors, errors
    for case, got in zip(jobs, outs):
        assert_parity(case, got)
    print("threads ok: %d calls" % (len(jobs) * REPEATS))


def test_first_calls_from_many_threads():
    r = subprocess.run([sys.executable, os.path.abspath(__file__)], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-4000:])
    assert "threads ok" in r.stdout


if __name__ == "__main__":
    _child()
