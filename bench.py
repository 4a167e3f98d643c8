"""Throughput of the dg GEMM path on GB300 (one JSON line on rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dg|reference]
                  [--workload NAME] [--configs default|all|none|NAME,...]

A step is one dg_gemm call: planning (cached), the tcgen05 main loop and the
fused alpha/beta/bias/GELU epilogue over one batch of synthetic inputs.  The
headline workload is the FP16 GEMM M = N = K = 4096 with D = 1.0*A.B + 0.5*C,
A, B ~ N(0,1)/sqrt(K), C ~ N(0,1) (seed 0).  Steps rotate over several input
sets whose total size is several times the 129 MB L2, so no step reads
operands another step left in L2.

After the headline (which also carries the end-to-end number through the
host-buffer call and the CPU oracle's rate), the same line holds a
`configs` object: every other configuration the library is measured on
(FP16 256^3, 2048^3 and 8192^3, INT8 4096^3, the thin M = 1 shapes, W4A16
at M = 16 and 2048, MXFP4 4096^3), each timed with the same K and W, with
its own value, roofline and clock record.  --configs none skips them.

--impl reference times the CPU oracle (fp64 definition of the same GEMM) on
the host cores, one bounded row sample of the same workload per step.

Multi-GPU (torchrun, one process per GPU): the GEMM does not shard, so each
rank runs an independent replica (weak scaling); value = all ranks' FLOPs /
the slowest rank's time.
"""

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "GEMM TFLOP/s (INT8 TOPS) and % of GB300 dense peak; GB/s vs HBM for M=1"
L2_BYTES = 129 * 1000 * 1000
RAMP_S = 0.2  # untimed clock ramp before the warm-up steps


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock and clock-event reasons of one GPU through NVML
    (read-only queries) in a background thread, about once a millisecond,
    from the ramp through the timed region; samples taken while the timed
    region runs are marked as such."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, index, period_s=0.0005):
        self.index, self.period = index, period_s
        self.samples = []  # (mhz, reasons, timed)
        self.ok = False
        self.timed = False
        self._stop = threading.Event()
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.handle)) != 0:
                return
            mx = ctypes.c_uint()
            self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx))  # 1 = SM
            self.max_mhz = int(mx.value)
            self.reasons_fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) \
                or self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = True
        except OSError:
            pass

    def _read(self):
        mhz, reasons = ctypes.c_uint(), ctypes.c_ulonglong()
        self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz))
        self.reasons_fn(self.handle, ctypes.byref(reasons))
        return int(mhz.value), int(reasons.value)

    def _run(self):
        while not self._stop.is_set():
            timed = self.timed
            m, r = self._read()
            self.samples.append((m, r, timed and self.timed))
            time.sleep(self.period)

    def mark_timed(self, on):
        self.timed = on

    def __enter__(self):
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self.t.join()

    def summary(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": "unavailable"}
        timed = [(m, r) for m, r, t in self.samples if t]
        # the median of the timed region's busy samples when it has a few,
        # else of every busy sample from the ramp on (a short timed region)
        use = timed if len(timed) >= 5 else [(m, r) for m, r, _ in self.samples]
        busy = [m for m, r in use if not (r & 0x1)] or [m for m, _ in use]
        seen = 0
        for _, r in use:
            seen |= r
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": self.max_mhz,
                "reasons": [n for b, n in self.REASONS.items() if seen & b and b != 0x1],
                "samples": len(self.samples), "samples_timed": len(timed),
                "over": "timed region" if use is timed else "ramp, warm-up and timed region",
                "source": "nvml"}


# --------------------------------------------------------------------------- helpers
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


KERNEL_SOURCES = {
    "gemm_tc_kernel": ("gemm_tc.cu", "tc_common.cuh", "ptx.cuh", "epilogue.cuh",
                           "internal.h"),
    "gemm_conv_tc_kernel": ("gemm_conv.cu", "tc_common.cuh", "ptx.cuh", "epilogue.cuh",
                            "internal.h"),
    "gemv_splitk_kernel": ("gemv.cu", "ptx.cuh", "epilogue.cuh", "internal.h"),
    "gemv_cluster_kernel": ("gemv.cu", "ptx.cuh", "epilogue.cuh", "internal.h"),
    "gemv_mma_kernel": ("gemv.cu", "ptx.cuh", "epilogue.cuh", "internal.h"),
    "skinny_w4a16_kernel": ("skinny.cu", "ptx.cuh", "epilogue.cuh", "internal.h"),
    "gemm_w4t_kernel": ("gemm_w4t.cu", "tc_common.cuh", "ptx.cuh", "epilogue.cuh", "internal.h"),
}


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kernel, ()):
        p = os.path.join(ROOT, "precision_matmul_dg_gb300", "csrc", f)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def recorded_capture(kernel, workload):
    """The committed ncu launch-list entry of a kernel on a workload (DRAM
    bytes per launch, the kernel's share of the step's launch time), if it
    was taken on the current sources of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(kernel, {}).get(workload)
    if not e or e.get("source_hash") != kernel_source_hash(kernel):
        return None
    return e


def recorded_traffic(kernel, workload):
    e = recorded_capture(kernel, workload)
    return e.get("dram_bytes_per_launch") if e else None


def workload_info(name):
    info = {
        "f16_4096": ("FP16 GEMM M=N=K=4096, D=1.0*A.B+0.5*C, A,B~N(0,1)/sqrt(K), C~N(0,1)",
                     "tensor"),
        "f16_2048": ("FP16 GEMM M=N=K=2048, D=1.0*A.B+0.5*C", "tensor"),
        "f16_8192": ("FP16 GEMM M=N=K=8192, D=1.0*A.B+0.5*C", "tensor"),
        "f16_256": ("FP16 GEMM M=N=K=256, A,B~U[-1,1)", "tensor"),
        "f16_256x4096x16384": ("FP16 GEMM M=256,N=4096,K=16384 (fewer tiles than SMs, long K), "
                               "D=1.0*A.B+0.5*C", "hbm"),
        "thin_1x4096x131072": ("FP16 GEMV M=1,N=4096,K=131072 split-K", "hbm"),
        "thin_1x256x12800": ("FP16 GEMV M=1,N=256,K=12800 split-K", "hbm"),
        "i8_4096": ("INT8 GEMM M=N=K=4096, A,B uniform int8, exact INT32 out", "tensor"),
        "w4a16_m16": ("W4A16 M=16,N=8960,K=1536, E2M1 weights x FP16, bias+erf-GELU", "hbm"),
        "w4a16_m256": ("W4A16 M=256,N=8960,K=1536, E2M1 weights x FP16, bias+erf-GELU",
                       "tensor"),
        "w4a16_m2048": ("W4A16 M=2048,N=8960,K=1536, E2M1 weights x FP16, bias+erf-GELU",
                        "tensor"),
        "qkv_1x128x4096_b96": ("96 FP16 GEMMs M=1,N=128,K=4096 in one strided-batched call "
                               "(QKV projections of 32 heads)", "hbm"),
        "moe_64x4096x2048": ("64 FP16 expert GEMMs N=4096, K=2048 with M uniform in 1..16, in one "
                             "grouped call (a mixture-of-experts layer)", "hbm"),
        "mxf4_4096": ("MXFP4 GEMM M=N=K=4096: FP16 activations quantized to MXFP4 (E2M1 codes, "
                      "one E8M0 scale per 32 along K) every step, times MXFP4 weights, "
                      "D=1.0*A.B+0.5*C, FP16 C/D", "tensor"),
    }
    return info[name]


def algorithmic_bytes(case):
    """Bytes the GEMM must move at least once: A, B, C (if read), bias, D."""
    mx = 0.5 + 1.0 / 32  # a code and a 32nd of a scale byte
    ea = {"f16": 2, "i8": 1, "mxf4": mx}[case.dtype_a]
    if case.a_fp16 is not None:
        ea = 2  # FP16 activations, quantized inside the step
    eb = {"f16": 2, "i8": 1, "e2m1": 0.5, "mxf4": mx}[case.dtype_b]
    ed = 4 if case.dtype_a == "i8" else 2
    if case.group_ms is not None:  # every expert's weights, its own rows of A and D
        rows = sum(case.group_ms)
        return int(case.batch * case.N * case.K * eb + rows * (case.K * ea + case.N * ed))
    b = case.M * case.K * ea + case.N * case.K * eb + case.M * case.N * ed
    if case.beta != 0:
        b += case.M * case.N * ed
    if case.bias is not None:
        b += case.N * 2
    return int(b * case.batch)


def kernel_name(plan, case):
    """The step's dominant kernel: the split-K GEMV, the tensor-core kernel
    (FP16; widened INT8 / E2M1 / MXFP4 operands; MXFP4 on the block-scaled
    MMA), the W4A16 kernel that widens the weights in tensor memory, or the
    converting kernel."""
    if plan["kernel_name"] == "gemv":
        # 2 .. 8 splits reduce inside a thread-block cluster
        return "gemv_cluster_kernel" if 2 <= plan["split_k"] <= 8 else "gemv_splitk_kernel"
    if plan["kernel_name"] == "skinny":
        return "skinny_w4a16_kernel"
    if plan["kernel_name"] == "gemv_mma":
        return "gemv_mma_kernel"
    if plan["kernel_name"] == "tc" and plan.get("swap_ab"):
        return "gemm_w4t_kernel"  # W4A16 with the weights widened in tensor memory
    if plan["kernel_name"] == "tc_widened" or case.dtype_a == "mxf4" or \
            (case.dtype_a == "f16" and case.dtype_b == "f16"):
        return "gemm_tc_kernel"
    return "gemm_conv_tc_kernel"


# --------------------------------------------------------------------------- GPU arm
class Workload:
    """One workload resident on the device: its input sets (rotated so that
    no step finds its operands in L2), its plan and the step that runs it."""

    def __init__(self, dg, name, dev, plan_index=0):
        self.dg, self.name, self.dev = dg, name, dev
        self.desc, self.bound = workload_info(name)
        base = self.base = workloads.WORKLOADS[name]()
        batch = base.batch
        self.out_dtype = torch.int32 if base.dtype_a == "i8" else torch.float16
        out_bytes = 4 if base.dtype_a == "i8" else 2
        self.out_shape = (batch, base.M, base.N) if batch > 1 else (base.M, base.N)
        self.is_mx = base.dtype_a == "mxf4"
        if self.is_mx:
            # the FP16 activations stand in the A slot; the step quantizes them
            base.A, base.scale_a = base.a_fp16, np.zeros((base.M, 1), np.uint8)
        set_bytes = base.A.nbytes + base.B.nbytes + batch * base.M * base.N * out_bytes
        if self.is_mx:
            set_bytes += base.scale_b.nbytes
        nsets = max(2, math.ceil(3 * L2_BYTES / set_bytes)) if set_bytes < 3 * L2_BYTES else 1
        self.nsets = min(nsets, 16)
        self.set_bytes = set_bytes
        self.A0 = torch.from_numpy(base.A).to(dev)
        self.B0 = torch.from_numpy(base.B).to(dev)
        C0 = (torch.from_numpy(base.C).to(dev) if base.C is not None else
              torch.zeros(*self.out_shape, dtype=self.out_dtype, device=dev))
        bias = torch.from_numpy(base.bias).to(dev) if base.bias is not None else None
        self.bias = bias
        self.SB0 = torch.from_numpy(base.scale_b).to(dev) if self.is_mx else None
        if self.is_mx:
            # the quantized activations: one buffer, rewritten by every step
            self.nblk = (base.K + 31) // 32
            self.ldq = self.nblk * 32
            self.QA = torch.empty((base.M, self.ldq // 2), dtype=torch.uint8, device=dev)
            self.QS = torch.empty((base.M, self.nblk), dtype=torch.uint8, device=dev)
        self.sets = []
        for s in range(self.nsets):
            # further sets: the same values with rows (problems, for a batch)
            # rotated (same distribution, different addresses), so no step finds
            # its operands in L2; scale rows move with their code rows
            sh = 37 * s
            roll = (lambda t: torch.roll(t, sh, 0).contiguous() if t is not None else None)
            self.sets.append((roll(self.A0), roll(self.B0), roll(C0), bias, roll(self.SB0)))
        cands = dg.plan_tiles(base.M, base.N, base.K, base.dtype_a, base.dtype_b, base.epilogue)
        plan = cands[min(plan_index, len(cands) - 1)]
        if base.group_ms is not None and base.dtype_a == "f16" and base.dtype_b == "f16" and \
                base.M <= 16:
            # an FP16 group whose largest M is at most 16 runs as one warp-MMA
            # GEMV launch over the problem table, whatever one problem's plan is
            plan = next(p for p in cands if p["kernel_name"] == "gemv_mma")
        self.plan = plan
        self.forced = plan if plan_index > 0 else None  # index 0: dg_gemm's own choice
        self.group_runs = None
        if base.group_ms is not None:
            # one prepared group per input set: the experts' rows of A and C
            # (the pointer arrays are built once, outside the timed steps)
            self.group_runs = [
                dg.prepare_grouped([A[g, :m] for g, m in enumerate(base.group_ms)],
                                   [B[g] for g in range(batch)],
                                   [C[g, :m] for g, m in enumerate(base.group_ms)],
                                   K=base.K, alpha=base.alpha, beta=base.beta,
                                   epilogue=base.epilogue)
                for A, B, C, _, _ in self.sets]

    def step(self, i, st):
        dg, base = self.dg, self.base
        if self.group_runs is not None:
            self.group_runs[i % self.nsets](st)
            return
        A, B, C, bias, SB = self.sets[i % self.nsets]
        if self.is_mx:
            dg.quantize_mxf4_raw(base.M, base.K, A, A.stride(0), self.QA, self.ldq, self.QS,
                                 self.nblk, stream=st)
            dg.gemm_mxf4(self.QA, self.QS, B, SB, C, base.K, bias=bias, alpha=base.alpha,
                         beta=base.beta, epilogue=base.epilogue, stream=st, plan=self.forced)
            return
        if base.batch > 1:
            dg.gemm_batched(A, B, C, K=base.K, bias=bias, alpha=base.alpha, beta=base.beta,
                            epilogue=base.epilogue, stream=st)
            return
        dg.gemm(A, B, C, K=base.K, bias=bias, alpha=base.alpha, beta=base.beta,
                epilogue=base.epilogue, stream=st, plan=self.forced)

    def work_unit(self):
        return work_unit(self.base, self.bound)


def time_workload(w, args, world, local, stream):
    """Ramp, W warm-up steps, then K timed steps between barriers and
    synchronizations (CUDA events on the launching stream).  Returns (total
    ms of the K steps, kernel launches inside them, the clock summary, the
    number of untimed ramp steps)."""
    dg, dev = w.dg, w.dev
    sampler = ClockSampler(local)
    with sampler:
        # An idle GPU needs a few tens of milliseconds of load before its
        # clocks settle: run the step untimed for RAMP_S before the warm-up.
        ramp_steps, t_ramp = 0, time.perf_counter()
        while time.perf_counter() - t_ramp < RAMP_S:
            for i in range(8):
                w.step(i, stream)
            torch.cuda.synchronize(dev)
            ramp_steps += 8
        for i in range(args.warmup):
            w.step(i, stream)
        dg.check_status(stream)
        torch.cuda.synchronize(dev)

        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        graph = None
        if args.graph:
            # The K timed steps captured once and replayed as one graph: the
            # launches run back to back with no host work between them.  Warm
            # up on the capture stream first: a split-K plan allocates its
            # per-stream workspace on first use, which must not happen
            # mid-capture.
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            for i in range(args.warmup):
                w.step(i, cap)
            torch.cuda.synchronize(dev)
            graph = torch.cuda.CUDAGraph()
            launches0 = dg.launch_count()
            with torch.cuda.graph(graph, stream=cap, capture_error_mode="thread_local"):
                for i in range(args.steps):
                    w.step(i, cap)
            launches = dg.launch_count() - launches0
            graph.replay()  # one untimed replay
            torch.cuda.synchronize(dev)
        else:
            launches0 = dg.launch_count()
        barrier(world)
        torch.cuda.synchronize(dev)
        sampler.mark_timed(True)
        t0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(args.steps):
                w.step(i, stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        sampler.mark_timed(False)
        barrier(world)
    if graph is None:
        launches = dg.launch_count() - launches0
    dg.check_status(stream)
    return t0.elapsed_time(t1), launches, sampler.summary(), ramp_steps


def roofline(w, kern_avg_ms, peaks, peak_src):
    """The dominant kernel's roofline: algorithmic FLOPs (tensor-bound) or
    bytes (HBM-bound) per launch over the launch's average duration."""
    base = w.base
    flops = base.flops()
    if w.bound == "tensor":
        achieved = flops / (kern_avg_ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "peak_source": "%s bf16 dense burst (fp16 runs at the bf16 rate)" % peak_src}
        # The same figure against the measured sustained rate (seconds of
        # back-to-back GEMMs under the power cap), for context: a timed region
        # of many launches runs under the same cap.  `frac` keeps the burst.
        if peaks.get("bf16_tflops_sustained"):
            roof["frac_of_sustained"] = round(achieved / peaks["bf16_tflops_sustained"], 4)
        if base.dtype_a == "i8":
            roof["unit"] = "TOPS"
            roof["peak_source"] += ("; INT8 runs on the FP16 tensor path (sm_103a has no "
                                    "integer tcgen05 MMA), so its denominator is the FP16 peak")
        if base.dtype_a == "mxf4":
            # block-scaled 4-bit operands: the FP4 dense peak, the measured
            # bf16 burst times the nominal FP4 / bf16 ratio (13.5 / 2.25)
            peak = round(peaks["bf16_tflops"] * 6.0, 1)
            roof.update(peak=peak, frac=round(achieved / peak, 4),
                        peak_source="%s bf16 dense burst x 6 (nominal FP4 / bf16 dense ratio)"
                                    % peak_src)
            if peaks.get("bf16_tflops_sustained"):
                roof["frac_of_sustained"] = round(achieved / (peaks["bf16_tflops_sustained"] * 6.0),
                                                  4)
    else:
        gbs = algorithmic_bytes(base) / (kern_avg_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                "frac": round(gbs / peak, 4), "peak_source": "%s copy bandwidth" % peak_src}
    kname = kernel_name(w.plan, base)
    roof["kernel"] = kname
    roof["kernel_avg_us"] = round(kern_avg_ms * 1e3, 2)
    roof["traffic"] = recorded_traffic(kname, w.name)
    steps = STEP_KERNELS.get(w.name)
    if steps:
        # A step of several launches: `achieved` divides by the whole step's
        # time; the committed launch list gives the dominant kernel's share
        cap = recorded_capture(kname, w.name)
        roof["step_kernels"] = steps
        roof["timed"] = "the whole step (every launch of it)"
        roof["share_of_step_ncu"] = cap.get("share_of_step") if cap else None
    roof["algorithmic_bytes"] = algorithmic_bytes(base)
    roof["algorithmic_flops"] = flops
    return roof


def plan_summary(plan):
    return {k: plan[k] for k in ("kernel_name", "m_tile", "n_tile", "k_tile", "split_k", "stages",
                                 "grid", "swap_ab")}


def measure_e2e(w, args, world, stream):
    """The same metric end to end: every step copies its inputs from pinned
    host memory to the device and its result back, inside the timed region."""
    dg, dev, base = w.dg, w.dev, w.base
    batch = base.batch
    hA = torch.from_numpy(base.A).pin_memory()
    hB = torch.from_numpy(base.B).pin_memory()
    hC = torch.from_numpy(base.C).pin_memory() if base.C is not None else None
    hbias = torch.from_numpy(base.bias).pin_memory() if base.bias is not None else None
    hD = torch.empty(*w.out_shape, dtype=w.out_dtype).pin_memory()
    call = "dg_gemm_host on pinned host buffers"
    h_scales = []
    if w.is_mx:
        # No host-buffer form of the MXFP4 call: the step copies the pinned
        # activations, codes, scales and C in, runs dg_quantize_mxf4 +
        # dg_gemm_mxf4 and copies D back.
        call = ("pinned host-to-device copies of the FP16 activations and the MXFP4 "
                "weights, dg_quantize_mxf4 + dg_gemm_mxf4, device-to-host copy")
        h_scales = [torch.from_numpy(base.scale_b).pin_memory()]
        dA, dB = torch.empty_like(w.A0), torch.empty_like(w.B0)
        dSB = torch.empty_like(w.SB0)
        dD = torch.empty(*w.out_shape, dtype=w.out_dtype, device=dev)
    if batch > 1:
        # The batched call takes device buffers: the step copies the pinned
        # inputs in, runs dg_gemm_strided_batched and copies D back.
        call = "pinned host-to-device copies, dg_gemm_strided_batched, device-to-host copy"
        dA, dB = torch.empty_like(w.A0), torch.empty_like(w.B0)
        dD = torch.empty(*w.out_shape, dtype=w.out_dtype, device=dev)
        dC = torch.empty_like(dD) if hC is not None else None
        dbias = torch.empty_like(w.bias) if hbias is not None else None
    if base.group_ms is not None:
        call = "pinned host-to-device copies, dg_gemm_grouped, device-to-host copy"
        dA, dB = torch.empty_like(w.A0), torch.empty_like(w.B0)
        dD = torch.empty(*w.out_shape, dtype=w.out_dtype, device=dev)
        e2e_group = dg.prepare_grouped([dA[g, :m] for g, m in enumerate(base.group_ms)],
                                       [dB[g] for g in range(batch)],
                                       [dD[g, :m] for g, m in enumerate(base.group_ms)],
                                       K=base.K, alpha=base.alpha, beta=base.beta,
                                       epilogue=base.epilogue)

    def e2e_step():
        if base.group_ms is not None:
            with torch.cuda.stream(stream):
                dA.copy_(hA, non_blocking=True)
                dB.copy_(hB, non_blocking=True)
                e2e_group(stream)
                hD.copy_(dD, non_blocking=True)
            return
        if w.is_mx:
            with torch.cuda.stream(stream):
                dA.copy_(hA, non_blocking=True)
                dB.copy_(hB, non_blocking=True)
                dSB.copy_(h_scales[0], non_blocking=True)
                if hC is not None:
                    dD.copy_(hC, non_blocking=True)
                dg.quantize_mxf4_raw(base.M, base.K, dA, dA.stride(0), w.QA, w.ldq, w.QS,
                                     w.nblk, stream=stream)
                dg.gemm_mxf4(w.QA, w.QS, dB, dSB, dD, base.K, bias=w.bias, alpha=base.alpha,
                             beta=base.beta, epilogue=base.epilogue, stream=stream)
                hD.copy_(dD, non_blocking=True)
            return
        if batch > 1:
            with torch.cuda.stream(stream):
                dA.copy_(hA, non_blocking=True)
                dB.copy_(hB, non_blocking=True)
                if dC is not None:
                    dC.copy_(hC, non_blocking=True)
                    dD.copy_(dC)
                if dbias is not None:
                    dbias.copy_(hbias, non_blocking=True)
                dg.gemm_batched(dA, dB, dD, K=base.K, bias=dbias, alpha=base.alpha,
                                beta=base.beta, epilogue=base.epilogue, stream=stream)
                hD.copy_(dD, non_blocking=True)
            return
        dg.gemm_host(hA, hB, hD, C=hC, K=base.K, bias=hbias, alpha=base.alpha, beta=base.beta,
                     epilogue=base.epilogue, dtype_b=base.dtype_b, stream=stream)

    e2e_steps = max(3, min(args.steps, 50))
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    work, unit = w.work_unit()
    value = sum_over_ranks(work * e2e_steps, world) / (e2e_ms * 1e-3) / 1e12
    return {"value": round(value, 2), "unit": unit,
            "h2d_bytes_per_step": int(hA.nbytes + hB.nbytes +
                                      sum(t.nbytes for t in h_scales) +
                                      (hC.nbytes if hC is not None else 0) +
                                      (hbias.nbytes if hbias is not None else 0)),
            "d2h_bytes_per_step": int(hD.nbytes),
            "call": "%s, %d steps" % (call, e2e_steps)}


def measure_config(dg, name, args, world, local, dev, stream, peaks, peak_src):
    """One further workload, timed exactly like the headline (same K and W,
    its own ramp, rotating inputs above L2): device-timed value, roofline and
    clocks.  Its buffers are freed before the next one."""
    w = Workload(dg, name, dev)
    total_ms, launches, clocks, _ = time_workload(w, args, world, local, stream)
    total_ms_max = max_over_ranks(total_ms, world)
    work, unit = w.work_unit()
    value = sum_over_ranks(work * args.steps, world) / (total_ms_max * 1e-3) / 1e12
    kern_avg_ms = total_ms / args.steps
    out = {"workload": w.desc, "value": round(value, 2), "unit": unit,
           "ms_per_step": round(total_ms_max / args.steps, 5),
           "kernel_avg_us": round(kern_avg_ms * 1e3, 2),
           "roofline": roofline(w, kern_avg_ms, peaks, peak_src),
           "plan": plan_summary(w.plan), "gpu_launches": int(launches), "clocks": clocks,
           "l2": ("%d rotating input sets, %.0f MB > L2" % (w.nsets, w.nsets * w.set_bytes / 1e6)
                  if w.nsets > 1 else "inputs larger than L2"),
           "timing": "eager back-to-back launches, CUDA events around the K steps"}
    if name in GRAPH_TOO and not args.graph:
        # A step of a few microseconds is bound by the host's launch path
        # when launched eagerly: the same K steps replayed from a CUDA graph
        # show the device time.
        gargs = argparse.Namespace(**vars(args))
        gargs.graph = True
        g_ms, _, g_clocks, _ = time_workload(w, gargs, world, local, stream)
        g_ms = max_over_ranks(g_ms, world)
        g_value = sum_over_ranks(work * args.steps, world) / (g_ms * 1e-3) / 1e12
        out["graph"] = {"value": round(g_value, 2), "unit": unit,
                        "kernel_avg_us": round(g_ms / args.steps * 1e3, 2),
                        "roofline": roofline(w, g_ms / args.steps, peaks, peak_src),
                        "clocks": g_clocks,
                        "timing": "one CUDA-graph replay of the K steps, CUDA events around it"}
    del w
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return out


def run_dg(args, world, rank, local):
    import precision_matmul_dg_gb300 as dg
    from precision_matmul_dg_gb300 import build as dg_build
    if rank == 0 or world > 1:
        dg_build.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()
    name = args.workload
    w = Workload(dg, name, dev, args.plan_index)
    base = w.base
    total_ms, launches, clocks, ramp_steps = time_workload(w, args, world, local, stream)
    # The K launches run back to back on one stream (eager or replayed from a
    # graph), each overlapping the previous one's drain; a launch's average
    # duration is the timed region over K.
    kern_avg_ms = total_ms / args.steps
    total_ms_max = max_over_ranks(total_ms, world)
    # Throughput unit: TFLOP/s (TOPS for INT8) for tensor-bound workloads,
    # algorithmic GB/s for the HBM-bound thin ones.
    work, unit = w.work_unit()
    value = sum_over_ranks(work * args.steps, world) / (total_ms_max * 1e-3) / 1e12
    e2e = measure_e2e(w, args, world, stream)
    roof = roofline(w, kern_avg_ms, peaks, peak_src)

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms_max / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": base.dtype_a,
        "data": "synthetic (seeded, recipe in workloads.py)",
        "config": {"workload": w.desc, "name": name, "M": base.M, "N": base.N, "K": base.K,
                   "batch": base.batch, "alpha": base.alpha, "beta": base.beta,
                   "epilogue": base.epilogue,
                   "ramp": "%d untimed steps (%.1f s) before the warm-up" % (ramp_steps, RAMP_S),
                   "timing": ("CUDA-graph replay of the K steps" if args.graph else
                              "eager back-to-back launches") +
                   ", CUDA events around the K steps, per launch = total / K",
                   "l2": "%d rotating input sets, %.0f MB > L2" % (w.nsets,
                                                                   w.nsets * w.set_bytes / 1e6)
                   if w.nsets > 1 else "inputs larger than L2",
                   "parallelism": "replicas" if world > 1 else "1 GPU",
                   "plan": plan_summary(w.plan),
                   "plan_note": ("the warp-MMA GEMV over the group's problem table (split-K "
                                 "chosen for the largest M)" if base.group_ms is not None else
                                 "the single problem's plan; a batched GEMV picks its split-K "
                                 "for the whole batch" if base.batch > 1 else "")},
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    del w
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    names = config_names(args, name)
    if names:
        line["configs"] = {}
        for n in names:
            line["configs"][n] = measure_config(dg, n, args, world, local, dev, stream, peaks,
                                                peak_src)
    return line


# The further workloads the default run measures after its headline, each
# with its own value, roofline and clocks: every configuration of the GEMM
# the library is measured on (square FP16 at three sizes and 256^3, INT8,
# the two thin M = 1 shapes, W4A16 at M = 16 and 2048, block-scaled FP4).
DEFAULT_CONFIGS = ("f16_256", "f16_2048", "f16_8192", "i8_4096", "thin_1x4096x131072",
                   "thin_1x256x12800", "w4a16_m16", "w4a16_m2048", "mxf4_4096")
# Steps of more than one launch (the dominant kernel last).
STEP_KERNELS = {"i8_4096": ["widen_dense_kernel", "gemm_tc_kernel"],
                "w4a16_m2048": ["widen_dense_kernel", "gemm_tc_kernel"],
                "mxf4_4096": ["quantize_mxf4_kernel", "gemm_tc_kernel"]}
# Workloads of a few microseconds a step, also timed as a CUDA-graph replay.
GRAPH_TOO = ("f16_256", "thin_1x256x12800", "w4a16_m16")


def config_names(args, headline):
    if args.configs == "none":
        return []
    names = DEFAULT_CONFIGS if args.configs == "default" else \
        tuple(sorted(workloads.WORKLOADS)) if args.configs == "all" else \
        tuple(n for n in args.configs.split(",") if n)
    for n in names:
        if n not in workloads.WORKLOADS:
            raise SystemExit("unknown workload in --configs: %s" % n)
    return [n for n in names if n != headline]


# --------------------------------------------------------------------------- CPU oracle
def work_unit(case, bound):
    """(work per whole problem, unit): FLOPs -> TFLOP/s (TOPS for INT8) for
    tensor-bound workloads, algorithmic bytes -> GB/s for HBM-bound ones; both
    scaled so that work / seconds / 1e12 is the value in that unit."""
    if bound == "hbm":
        return algorithmic_bytes(case) * 1e3, "GB/s"
    return case.flops(), ("TOPS" if case.dtype_a == "i8" else "TFLOP/s")


def oracle_rows(oracle, case, rows):
    """The oracle's D on the given rows of a single-problem case."""
    kw = dict(C=case.C, bias=case.bias, alpha=case.alpha, beta=case.beta,
              epilogue=case.epilogue, rows=rows)
    if case.dtype_a == "mxf4" and case.a_fp16 is not None:
        # quantize the activation rows, then multiply
        codes, scales = oracle.mxfp4_quantize(case.a_fp16[rows], case.K)
        kw.update(rows=None, C=case.C[rows] if case.C is not None else None)
        return oracle.gemm_mx_reference(oracle.pack_e2m1(codes), scales, case.B, case.scale_b,
                                        case.K, **kw)
    if case.dtype_a == "mxf4":
        return oracle.gemm_mx_reference(case.A, case.scale_a, case.B, case.scale_b, case.K, **kw)
    return oracle.gemm_reference(case.A, case.B, case.K, case.dtype_a, case.dtype_b, **kw)


def oracle_sample_rate(case, budget_s, rows_per_call, bound="tensor"):
    """Times the oracle (fp64 definition) on row samples of `case` for about
    budget_s seconds; returns (value in the metric's unit, unit, seconds,
    rows done)."""
    import oracle
    rng = np.random.default_rng(0)
    done_rows, t_total = 0, 0.0
    if case.batch > 1:  # whole problems, chosen at random
        total_rows = sum(case.group_ms) if case.group_ms is not None else case.M * case.batch
        while t_total < budget_s and done_rows < total_rows:
            z = int(rng.integers(case.batch))
            m = case.group_ms[z] if case.group_ms is not None else case.M
            t = time.perf_counter()
            oracle.gemm_reference(case.A[z][:m], case.B[z], case.K, case.dtype_a, case.dtype_b,
                                  alpha=case.alpha, beta=case.beta, epilogue=case.epilogue)
            t_total += time.perf_counter() - t
            done_rows += m
        work, unit = work_unit(case, bound)
        return work * done_rows / total_rows / t_total / 1e12, unit, t_total, done_rows
    while t_total < budget_s and done_rows < 64 * case.M:
        rows = rng.choice(case.M, size=min(rows_per_call, case.M), replace=False)
        t = time.perf_counter()
        oracle_rows(oracle, case, rows)
        t_total += time.perf_counter() - t
        done_rows += len(rows)
    work, unit = work_unit(case, bound)
    return work * done_rows / case.M / t_total / 1e12, unit, t_total, done_rows


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args):
    name = args.workload
    desc, _ = workload_info(name)
    case = workloads.WORKLOADS[name]()
    rows = max(1, min(case.M, 64))
    import oracle
    rng = np.random.default_rng(1)
    done = []  # rows of each whole-problem step

    def step():
        if case.batch > 1:  # one whole problem per step
            z = int(rng.integers(case.batch))
            m = case.group_ms[z] if case.group_ms is not None else case.M
            done.append(m)
            oracle.gemm_reference(case.A[z][:m], case.B[z], case.K, case.dtype_a, case.dtype_b,
                                  alpha=case.alpha, beta=case.beta, epilogue=case.epilogue)
            return
        r = rng.choice(case.M, size=rows, replace=False)
        oracle_rows(oracle, case, r)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t
    work, unit = work_unit(case, workload_info(name)[1])
    if case.batch > 1:
        total_rows = sum(case.group_ms) if case.group_ms is not None else case.M * case.batch
        value = work * sum(done[args.warmup:]) / total_rows / dt / 1e12
        sample = "one random problem of the %d per step (%s)" % (case.batch, name)
    else:
        value = work * rows / case.M * args.steps / dt / 1e12
        sample = "%d random rows of the %dx%dx%d product per step (%s)" % (rows, case.M, case.N,
                                                                          case.K, name)
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value, "unit": unit, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, recipe in workloads.py)",
        "config": {"workload": desc, "name": name, "M": case.M, "N": case.N, "K": case.K,
                   "alpha": case.alpha, "beta": case.beta, "epilogue": case.epilogue},
        "cpu_baseline": {"value": value, "unit": unit, "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="dg", choices=["dg", "reference"])
    ap.add_argument("--workload", default="f16_4096")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--configs", default="default",
                    help="further workloads measured after the headline into the line's "
                         "`configs` object: default (every measured configuration), all, "
                         "none, or a comma-separated list of names")
    ap.add_argument("--plan-index", type=int, default=0,
                    help="run the planner's i-th ranked candidate instead of its first")
    ap.add_argument("--graph", action="store_true",
                    help="time one CUDA-graph replay of the K steps (no host work between "
                         "launches); per-launch time = total / K")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        import subprocess
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               "--nproc-per-node", str(args.gpus), "--master-addr", "127.0.0.1",
               "--master-port", "29511", os.path.abspath(__file__)] + sys.argv[1:]
        sys.exit(subprocess.call(cmd))

    world, rank, local = dist_setup()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    line = run_dg(args, world, rank, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            case = workloads.WORKLOADS[args.workload]()
            v, u, secs, rows = oracle_sample_rate(case, budget_s=10.0, rows_per_call=256,
                                                  bound=workload_info(args.workload)[1])
            line["cpu_baseline"] = {
                "value": v, "unit": u, "cores": cpu_cores(), "kind": "oracle",
                "sample": "%d rows of the %s%dx%dx%d product in %.1f s (fp64 numpy BLAS, "
                          "default threads)" % (rows, "%d x " % case.batch if case.batch > 1
                                                else "", case.M, case.N, case.K, secs)}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
