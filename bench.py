"""Benchmark of the SVDQuant W4A4 linear layer (svdq_linear_forward) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload flux_mlp_up] [--impl reference]

One step = one pass of the whole hot path (kernel 1: smoothing + NVFP4 quantisation +
down-projection; kernel 2: block-scaled FP4 tensor-core GEMM + up-projection + bias) over
one batch of synthetic FLUX-shaped activations already resident in HBM.  L2 is flushed
(a 256 MiB read that leaves clean lines) before every timed step, outside the timed events.
Prints one JSON line.  At one GPU the line also carries a `sweep` of every timed point of the
FLUX-shaped scope (QKV, MLP up/down, the output projection over tokens and ranks): kernel-by-
kernel medians with cold and warm L2, the fractions of the FP4 and HBM rooflines and the
low-rank branch's overhead.

Under torchrun (N > 1) every rank runs its own replica on its own GPU with its own batch
(the layer shards over tokens with no exchange): weak scaling, time = max over ranks.

--impl reference times the CPU oracle (the plain numpy restatement of the method) on the
host cores over all M rows of the same workload (fewer rows per step only if K steps of the
whole workload would exceed about three minutes), in the same metric.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from w4a4_rank_corrected_e2m1_b300 import synthetic  # noqa: E402

METRIC = "fused SVDQuant W4A4 linear TFLOPS & tokens/s at FLUX shapes; % of FP4 roofline"
FP4_OVER_BF16 = 13.5 / 2.25          # nominal dense FP4 : BF16 tensor ratio on B300

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch, from the ncu
# captures summarised under profiles/, keyed by the workload and by a hash of the kernel's
# sources at capture time: a kernel edited since then reports null traffic.
NCU_TRAFFIC = {
    ("flux_mlp_up", "k1_actquant"): ("6d066dcbfff4071a", 28570624.0 + 0.0),
    ("flux_mlp_up", "k2_fp4gemm"): ("d43e44583deda194", 36343552.0 + 64710400.0),
    ("flux_mod", "awq_gemv"): ("11f7be6295e75b32", 35478016.0 + 0.0),
}
KERNEL_SOURCES = {
    "k1_actquant": ["k1_actquant.cu", "nvfp4_block.cuh", "ptx.cuh", "svdq_internal.h"],
    "k2_fp4gemm": ["k2_fp4gemm.cu", "nvfp4_block.cuh", "ptx.cuh", "svdq_internal.h"],
    "awq_gemv": ["awq_gemv.cu", "ptx.cuh", "svdq_internal.h"],
}


def kernel_source_hash(kernel):
    """Hash of a kernel's sources with comments and whitespace removed: a code change alters it,
    a comment edit does not."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "w4a4_rank_corrected_e2m1_b300", "csrc", f)) as fh:
            txt = fh.read()
        txt = re.sub(r"/\*.*?\*/", " ", txt, flags=re.S)
        txt = re.sub(r"//[^\n]*", " ", txt)
        h.update(" ".join(txt.split()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload, kernel):
    """Captured DRAM bytes per launch, or None if absent or the kernel's code changed since."""
    entry = NCU_TRAFFIC.get((workload, kernel))
    if entry is None:
        return None
    return entry[1] if kernel_source_hash(kernel) == entry[0] else None


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="flux_mlp_up",
                    choices=sorted(synthetic.WORKLOADS) + [synthetic.MLP_PAIR.name])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="time the headline workload only")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6400.0, 1800.0, "fallback"


def batch_seeds(rank, nbuf):
    """Seeds of the activation batches a rank cycles through: disjoint across ranks, so the
    replicas work on different tokens."""
    return [1000 * rank + i for i in range(nbuf)]


def max_over_ranks(values, world, device):
    """Element-wise maximum over ranks of per-rank floats: the job's time is its slowest rank's."""
    if world == 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def job_rate(units_per_rank, world, seconds):
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world / seconds


def workload_flops(w, rows=None):
    M = w.M if rows is None else rows
    return 2.0 * M * w.N * w.K + 2.0 * M * w.K * w.rank + 2.0 * M * w.rank * w.N


# ------------------------------------------------------------------ CPU oracle timing
def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except ImportError:
        return len(os.sched_getaffinity(0))


def oracle_sample(w, d, p, budget_s=10.0):
    """Time the oracle forward on a bounded sample of rows of the workload, given a packed
    layer p; returns (TFLOP/s, rows, seconds)."""
    from oracle import svdquant as sq
    rows = 16
    while True:
        t0 = time.perf_counter()
        sq.forward(d["X"][:rows], p)
        dt = time.perf_counter() - t0
        if dt > budget_s / 3 or rows >= w.M:
            break
        rows = min(w.M, rows * 4)
    return workload_flops(w, rows) / dt / 1e12, rows, dt


def run_reference(args, w, budget_s=180.0):
    """The oracle forward on the host cores, every step over the workload's M rows (like the
    cpu_baseline leg of the GPU arm), unless K + 1 such steps would exceed the budget: then each
    step takes an equal share of the rows, at least 512."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    d = synthetic.make(w)
    from oracle import svdquant as sq
    p = sq.pack(d["W"], d["bias"], w.rank, Xcal_bits=d["X"])
    t0 = time.perf_counter()
    sq.forward(d["X"], p)                                 # warm-up over all rows, also the estimate
    t_full = time.perf_counter() - t0
    rows = w.M
    if t_full * (args.steps + 1) > budget_s:
        rows = max(min(w.M, 512), int(w.M * budget_s / (t_full * (args.steps + 1))))
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        sq.forward(d["X"][:rows], p)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    val = workload_flops(w, rows) * args.steps / tot / 1e12
    threads = blas_threads()
    sample = (f"{rows} of {w.M} token rows per step, {args.steps} steps after one warm-up step over all rows "
              f"(oracle forward; the layer packed once by the oracle)")
    out = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": 1, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "M": w.M, "K": w.K, "N": w.N, "rank": w.rank},
        "tokens_per_s": rows * args.steps / tot,
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)),
                         "threads": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ clocks
class _Nvml:
    """The few NVML calls the sampler needs, through ctypes on the driver's libnvidia-ml."""

    CLOCK_SM = 1

    def __init__(self, cuda_index):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        n = ctypes.c_uint()
        self.lib.nvmlDeviceGetCount_v2(ctypes.byref(n))
        idx = cuda_index
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        if n.value == 1:
            idx = 0
        elif vis and all(v.strip().isdigit() for v in vis.split(",")):
            idx = int(vis.split(",")[cuda_index])
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def max_sm(self):
        v = self.ct.c_uint()
        return v.value if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, self.ct.byref(v)) == 0 else None

    def sample(self):
        sm, rs = self.ct.c_uint(), self.ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, self.ct.byref(sm)) != 0:
            return None
        if self.reasons_fn(self.h, self.ct.byref(rs)) != 0:
            return None
        return sm.value, rs.value


class Clocks:
    """SM clock and throttle reasons sampled during the timed region.

    NVML (the library nvidia-smi reads, through ctypes) polled about every half millisecond
    from a thread, so that short timed regions still get samples; falls back to
    `nvidia-smi --query-gpu ... -lms 100`."""

    REASONS = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
               "sw_power_cap": 0x4, "hw_power_brake_slowdown": 0x80}

    def __init__(self, device_index):
        import threading
        self.samples = []
        self.stop_ev = threading.Event()
        self.proc = None
        try:
            nv = _Nvml(device_index)
            self.max_mhz = nv.max_sm()

            def run():
                while not self.stop_ev.is_set():
                    x = nv.sample()
                    if x is not None:
                        self.samples.append(x)
                    time.sleep(0.0005)
            self.thread = threading.Thread(target=run, daemon=True)
            self.thread.start()
        except Exception:
            self.thread = None
            self.max_mhz = None
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(device_index), "--query-gpu=clocks.sm,clocks.max.sm,"
                     "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=self.f, stderr=subprocess.DEVNULL)
            except Exception:
                self.proc = None

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        if self.thread is not None:
            self.stop_ev.set()
            self.thread.join()
            out["source"] = "nvml"
            if self.samples:
                sm = [x[0] for x in self.samples]
                mask = 0
                for x in self.samples:
                    mask |= x[1]
                out.update(sm_mhz=statistics.median(sm), samples=len(sm),
                           reasons=sorted(n for n, b in self.REASONS.items() if mask & b))
            return out
        if self.proc is not None:
            self.proc.terminate()
            self.proc.wait()
            self.f.flush()
            rows = [[x.strip() for x in line.split(",")] for line in open(self.f.name)]
            os.unlink(self.f.name)
            sm = [float(r[0]) for r in rows if r and r[0].replace(".", "").isdigit()]
            mx = [float(r[1]) for r in rows if len(r) > 1 and r[1].replace(".", "").isdigit()]
            out.update(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(mx) if mx else None,
                       samples=len(sm), source="nvidia-smi")
        return out


# ------------------------------------------------------------------ GPU arm
class L2Flush:
    """Evicts L2 between timed steps by reading (not writing) a 256 MiB buffer that was written
    once at set-up: L2 is left holding clean lines, so the next kernel's reads evict them for
    free instead of paying the write-back of dirty lines inside its own timed window."""

    def __init__(self, torch):
        self.torch = torch
        self.buf = torch.ones(64 << 20, dtype=torch.int32, device="cuda")
        self.acc = torch.empty((), dtype=torch.int32, device="cuda")

    def __call__(self):
        # int32 in and out: one reduction kernel, no widening copy of the buffer first
        self.torch.sum(self.buf, dim=0, dtype=self.torch.int32, out=self.acc)


def k1_bytes(M, K, rank):
    """Algorithmic HBM bytes of kernel 1: X read, codes, scales and T written, L1 and 1/lambda."""
    return M * K * 2 + M * K // 2 + M * K // 16 + M * rank * 2 + K * rank * 2 + K * 4


class Point:
    """One workload on one GPU: the packed layer at its rank and at rank 0, resident inputs and
    outputs, and the kernel-by-kernel buffers."""

    def __init__(self, torch, svdq, w, device, rank_seed=0, nbuf=1):
        self.torch, self.w = torch, w
        d = synthetic.make(w)
        t0 = time.perf_counter()
        self.layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], M_max=w.M, device=device)
        self.pack_s = time.perf_counter() - t0
        self.layer0 = svdq.Layer(d["W"], 0, bias=d["bias"], Xcal=d["X"], M_max=w.M, device=device)
        self.d = d
        M, K, N = w.M, w.K, w.N
        self.Xs = [torch.from_numpy(synthetic.make_x(w, M, seed=sd).view(np.int16)).cuda()
                   for sd in batch_seeds(rank_seed, nbuf)]
        self.Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        self.codes = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
        self.scales = torch.empty(svdq.scales_bytes(M, K), dtype=torch.uint8, device="cuda")
        self.T = torch.empty((M, max(self.layer.info.r_pad, 8)), dtype=torch.int16, device="cuda")

    def close(self):
        self.layer.close()
        self.layer0.close()


def time_events(torch, stream, body, reps, warm, flush, marks):
    """Run body(i, ev) reps + warm times; ev is a list of `marks` events body records on
    `stream`.  With `flush`, L2 is flushed before every iteration, outside the events.
    Returns the per-iteration lists of consecutive event gaps (ms) of the timed iterations."""
    for i in range(warm):
        if flush:
            flush()
        body(i, None)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(marks)] for _ in range(reps)]
    for i in range(reps):
        if flush:
            flush()
        body(i, evs[i])
    torch.cuda.synchronize()
    return [[e[j].elapsed_time(e[j + 1]) for j in range(marks - 1)] for e in evs]


def measure_point(torch, pt, stream, reps, warm, flush):
    """Medians (microseconds) of the forward and of kernel 1 and kernel 2 run one at a time, at
    the point's rank and at rank 0, with L2 flushed before every run (cold) and without (warm)."""
    lay, lay0, M, nb = pt.layer, pt.layer0, pt.w.M, len(pt.Xs)

    def fwd(layer):
        def body(i, ev):
            if ev:
                ev[0].record(stream)
            layer.forward(pt.Xs[i % nb], pt.Y, M, stream)
            if ev:
                ev[1].record(stream)
        return body

    def split(layer):
        def body(i, ev):
            if ev:
                ev[0].record(stream)
            layer.quantize_act(pt.Xs[i % nb], M, pt.codes, pt.scales, pt.T, stream)
            if ev:
                ev[1].record(stream)
            layer.gemm_quantized(pt.codes, pt.scales, pt.T, pt.Y, M, stream)
            if ev:
                ev[2].record(stream)
        return body

    out = {}
    for mode, fl in (("cold", flush), ("warm", None)):
        f = time_events(torch, stream, fwd(lay), reps, warm, fl, 2)
        k = time_events(torch, stream, split(lay), reps, warm, fl, 3)
        k0 = time_events(torch, stream, split(lay0), reps, warm, fl, 3)
        med = lambda rows, j: 1e3 * statistics.median(r[j] for r in rows)
        out[mode] = {"fwd_us": med(f, 0), "k1_us": med(k, 0), "k2_us": med(k, 1),
                     "k1_rank0_us": med(k0, 0), "k2_rank0_us": med(k0, 1)}
    lay.check_error()
    lay0.check_error()
    return out


def point_summary(w, t, hbm, fp4_peak):
    """Per-point figures of the scope table's measurement row, from measure_point's times."""
    c = t["cold"]
    lowrank = ((c["k1_us"] + c["k2_us"]) - (c["k1_rank0_us"] + c["k2_rank0_us"])) / c["k2_rank0_us"]
    return {
        "M": w.M, "K": w.K, "N": w.N, "rank": w.rank,
        "cold_l2": {k: round(v, 2) for k, v in c.items()},
        "warm_l2": {k: round(v, 2) for k, v in t["warm"].items()},
        "tflops": workload_flops(w) / (c["fwd_us"] * 1e-6) / 1e12,
        "tokens_per_s": w.M / (c["fwd_us"] * 1e-6),
        "frac_fp4_k2": 2.0 * w.M * w.N * w.K / (c["k2_us"] * 1e-6) / 1e12 / fp4_peak,
        "frac_hbm_k1": k1_bytes(w.M, w.K, w.rank) / (c["k1_us"] * 1e-6) / 1e9 / hbm,
        "lowrank_overhead": lowrank,
    }


def measure_int4(torch, svdq, w, pt, stream, flush, bf16_peak, reps=50, warm=5):
    """The INT4 variant of the same layer (svdq_int4_forward and its activation kernel alone) on
    the headline workload: medians with cold and warm L2.  Its GEMM runs bf16 warp MMAs on
    unpacked INT4 codes, so the fraction is against the measured bf16 tensor peak."""
    M, K = w.M, w.K
    layer = svdq.Int4Layer(pt.d["W"], w.rank, bias=pt.d["bias"], Xcal=pt.d["X"], M_max=M)
    codes = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((K // 64, svdq.int4_scale_ld(M)), dtype=torch.float32, device="cuda")
    T = torch.empty((M, max(layer.r_pad, 8)), dtype=torch.int16, device="cuda")
    nb = len(pt.Xs)

    def fwd(i, ev):
        if ev:
            ev[0].record(stream)
        layer.forward(pt.Xs[i % nb], pt.Y, M, stream)
        if ev:
            ev[1].record(stream)

    def k1(i, ev):
        if ev:
            ev[0].record(stream)
        layer.quantize_act(pt.Xs[i % nb], M, codes, scales, T, stream)
        if ev:
            ev[1].record(stream)

    out = {}
    for mode, fl in (("cold_l2", flush), ("warm_l2", None)):
        f = time_events(torch, stream, fwd, reps, warm, fl, 2)
        k = time_events(torch, stream, k1, reps, warm, fl, 2)
        out[mode] = {"fwd_us": round(1e3 * statistics.median(r[0] for r in f), 2),
                     "k1_us": round(1e3 * statistics.median(r[0] for r in k), 2)}
    layer.check_error()
    layer.close()
    t = out["cold_l2"]["fwd_us"] * 1e-6
    tflops = workload_flops(w) / t / 1e12
    out.update(workload=w.name, tflops=tflops, tokens_per_s=M / t, frac_bf16_peak=tflops / bf16_peak,
               note="INT4 groups of 64 (float32 scales); GEMM on bf16 warp MMAs over unpacked codes; "
                    "fraction of the measured bf16 tensor peak")
    return out


def measure_mlp_pair(torch, svdq, pw, stream, flush, reps=50, warm=5):
    """The MLP pair (up layer, GELU, down layer) run unfused (svdq_linear_forward, svdq_gelu_bf16,
    svdq_linear_forward) and fused (svdq_mlp_forward: the up layer's kernel 2 writes the down
    layer's quantised input); medians with cold and warm L2, and the parts of each."""
    up_w, dn_w = pw.up, pw.down
    M, K, Nu, N = up_w.M, up_w.K, up_w.N, dn_w.N
    d = synthetic.make(up_w)
    up = svdq.Layer(d["W"], up_w.rank, bias=d["bias"], Xcal=d["X"], M_max=M)
    X = torch.from_numpy(d["X"].view(np.int16)).cuda()
    Yup = torch.empty((M, Nu), dtype=torch.bfloat16, device="cuda")
    G = torch.empty_like(Yup)
    up.forward(X, Yup, M, stream)
    svdq.gelu_bf16(Yup, G, M * Nu, stream)
    torch.cuda.synchronize()
    # the down layer calibrated on its real input (a sample of rows of G)
    Gcal = G[: min(M, 1024)].view(torch.int16).cpu().numpy().view(np.uint16)
    wd = synthetic.make_weights(dn_w)
    down = svdq.Layer(wd["W"], dn_w.rank, bias=wd["bias"], Xcal=Gcal, M_max=M)
    mlp = svdq.Mlp(up, down, M)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    codes = torch.empty((M, Nu // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty(svdq.scales_bytes(M, Nu), dtype=torch.uint8, device="cuda")
    T = torch.empty((M, max(down.info.r_pad, 8)), dtype=torch.int16, device="cuda")

    def unfused(i, ev):
        if ev:
            ev[0].record(stream)
        up.forward(X, Yup, M, stream)
        if ev:
            ev[1].record(stream)
        svdq.gelu_bf16(Yup, G, M * Nu, stream)
        if ev:
            ev[2].record(stream)
        down.forward(G, Y, M, stream)
        if ev:
            ev[3].record(stream)

    def fused(i, ev):
        if ev:
            ev[0].record(stream)
        mlp.up_quantize(X, M, codes, scales, T, stream)
        if ev:
            ev[1].record(stream)
        down.gemm_quantized(codes, scales, T, Y, M, stream)
        if ev:
            ev[2].record(stream)

    def whole(i, ev):
        if ev:
            ev[0].record(stream)
        mlp.forward(X, Y, M, stream)
        if ev:
            ev[1].record(stream)

    med = lambda rows, j: round(1e3 * statistics.median(r[j] for r in rows), 2)
    out = {}
    for mode, fl in (("cold_l2", flush), ("warm_l2", None)):
        u = time_events(torch, stream, unfused, reps, warm, fl, 4)
        f = time_events(torch, stream, fused, reps, warm, fl, 3)
        h = time_events(torch, stream, whole, reps, warm, fl, 2)
        out[mode] = {"unfused_us": round(1e3 * statistics.median(sum(r) for r in u), 2),
                     "unfused_up_us": med(u, 0), "unfused_gelu_us": med(u, 1), "unfused_down_us": med(u, 2),
                     "fused_us": med(h, 0), "fused_up_quantize_us": med(f, 0), "fused_down_gemm_us": med(f, 1)}
    mlp.check_error()
    flops = 2.0 * M * Nu * K + 2.0 * M * N * Nu + 2.0 * M * up_w.rank * (K + Nu) + 2.0 * M * dn_w.rank * (Nu + N)
    c = out["cold_l2"]
    out.update(workload=pw.name, M=M, K=K, N_up=Nu, N=N, ranks=[up_w.rank, dn_w.rank],
               tflops_fused=flops / (c["fused_us"] * 1e-6) / 1e12,
               tflops_unfused=flops / (c["unfused_us"] * 1e-6) / 1e12,
               speedup=c["unfused_us"] / c["fused_us"],
               hbm_bytes_avoided=4 * M * Nu * 2,
               note="unfused = up forward, GELU kernel, down forward; fused = up kernels 1 and 2 with the "
                    "GELU + next-layer quantiser epilogue and the T reduction, then the down layer's kernel 2; "
                    "avoided: Y_up written, GELU's read and write, the down kernel 1's read of G")
    mlp.close()
    down.close()
    up.close()
    return out


def run_ours(args, w):
    import torch
    import torch.distributed as dist
    from w4a4_rank_corrected_e2m1_b300 import svdq

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    hbm, bf16, src = peaks()
    fp4_peak = bf16 * FP4_OVER_BF16
    # distinct activation batches per step (rank-specific seeds), resident in HBM
    pt = Point(torch, svdq, w, local, rank_seed=rank, nbuf=4)
    layer, M, K, N = pt.layer, w.M, w.K, w.N
    stream = torch.cuda.current_stream()
    flush = L2Flush(torch)

    # ---- the headline: K timed forwards, L2 flushed before each (outside the events)
    for i in range(args.warmup):
        flush()
        layer.forward(pt.Xs[i % 4], pt.Y, M, stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device())
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush()
        ev[i][0].record(stream)
        layer.forward(pt.Xs[i % 4], pt.Y, M, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    torch.cuda.synchronize()
    fwd_ms = [a.elapsed_time(b) for a, b in ev]
    layer.check_error()

    # ---- kernel by kernel, at the layer's rank and at rank 0 (cold and warm L2)
    reps = max(100, args.steps)
    t = measure_point(torch, pt, stream, reps, 10, flush)

    # ---- end to end through the pipelined host-buffer entry point: every step uploads its own
    # X from pinned host memory and downloads its Y; uploads, kernels and downloads of
    # neighbouring steps overlap (two staging slots); host wall time over the whole batch
    layer.reserve(M, host_staging=2)
    Xh = [torch.from_numpy(synthetic.make_x(w, M, seed=77 + 2 * rank + i).view(np.int16)).pin_memory()
          for i in range(2)]
    Yh = [torch.empty((M, N), dtype=torch.int16).pin_memory() for _ in range(2)]
    n_e2e = max(4, args.steps // 2)
    layer.forward_host_batch([Xh[i % 2] for i in range(max(2, args.warmup))],
                             [Yh[i % 2] for i in range(max(2, args.warmup))], M, stream)
    barrier()
    e2e_t = []
    for _ in range(3):
        t0 = time.perf_counter()
        layer.forward_host_batch([Xh[i % 2] for i in range(n_e2e)], [Yh[i % 2] for i in range(n_e2e)], M, stream)
        e2e_t.append((time.perf_counter() - t0) / n_e2e)
    barrier()

    ms_step, e2e_med = max_over_ranks([sum(fwd_ms) / len(fwd_ms), statistics.median(e2e_t)], world, "cuda")

    # ---- every other timed point of the scope table (one GPU only: the scaling runs time the
    # headline alone)
    sweep = {}
    int4 = None
    if world == 1 and not args.no_sweep:
        int4 = measure_int4(torch, svdq, w, pt, stream, flush, bf16)
        sweep[synthetic.MLP_PAIR.name] = measure_mlp_pair(torch, svdq, synthetic.MLP_PAIR, stream, flush)
        torch.cuda.empty_cache()
        for sw in synthetic.SWEEP:
            if sw.name == w.name:
                sweep[sw.name] = point_summary(sw, t, hbm, fp4_peak)
                continue
            p2 = Point(torch, svdq, sw, local)
            sweep[sw.name] = point_summary(sw, measure_point(torch, p2, stream, 100, 10, flush), hbm, fp4_peak)
            p2.close()
            del p2
            torch.cuda.empty_cache()

    if rank == 0:
        flops = workload_flops(w)
        tflops = job_rate(flops, world, ms_step * 1e-3) / 1e12
        c = t["cold"]
        t_k1, t_k2 = c["k1_us"] * 1e-3, c["k2_us"] * 1e-3
        k2_fp4_flops = 2.0 * M * N * K
        k2_achieved = k2_fp4_flops / (t_k2 * 1e-3) / 1e12
        kb = k1_bytes(M, K, w.rank)
        head = point_summary(w, t, hbm, fp4_peak)
        out = {
            "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "nvfp4(e2m1,e4m3)+bf16, f32 accumulate", "data": "synthetic",
            "config": {"workload": w.name, "M": M, "K": K, "N": N, "rank": w.rank, "per_gpu_tokens": M,
                       "l2": "flushed before every timed step (a 256 MiB read, outside the timed events)",
                       "parallelism": f"replicas x{world} (token shards, no collective)"},
            "tokens_per_s": job_rate(M, world, ms_step * 1e-3),
            "kernels_ms": {"k1_actquant": t_k1, "k2_fp4gemm": t_k2},
            "roofline": {"bound": "tensor", "kernel": "k2_fp4gemm", "achieved": k2_achieved, "peak": fp4_peak,
                         "unit": "TFLOP/s", "frac": k2_achieved / fp4_peak,
                         "traffic": ncu_traffic(w.name, "k2_fp4gemm"), "traffic_unit": "bytes per launch (ncu)",
                         "algorithmic_flop": k2_fp4_flops,
                         "peak_source": f"{src} bf16 {bf16} TFLOP/s x {FP4_OVER_BF16:g} (nominal FP4:BF16)"},
            "roofline_k1": {"bound": "hbm", "kernel": "k1_actquant", "achieved": kb / (t_k1 * 1e-3) / 1e9,
                            "peak": hbm, "unit": "GB/s", "frac": kb / (t_k1 * 1e-3) / 1e9 / hbm,
                            "traffic": ncu_traffic(w.name, "k1_actquant"), "traffic_unit": "bytes per launch (ncu)",
                            "algorithmic_bytes": kb},
            "lowrank": {"rank": w.rank, "k1_us": c["k1_us"], "k2_us": c["k2_us"],
                        "k1_rank0_us": c["k1_rank0_us"], "k2_rank0_us": c["k2_rank0_us"],
                        "overhead_frac_of_plain_4bit_gemm": head["lowrank_overhead"],
                        "formula": "[t(K1) + t(K2)] - [t(K1, r=0) + t(K2, r=0)], over t(K2, r=0); cold L2, medians"},
            "e2e": {"value": job_rate(flops, world, e2e_med) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": M * K * 2, "d2h_bytes_per_step": M * N * 2,
                    "ms_per_step": e2e_med * 1e3, "steps_per_call": n_e2e,
                    "api": "svdq_linear_forward_host_batch (pipelined, two staging slots)"},
            "gpu_launches": 2 * args.steps,
            "clocks": clk,
            "pack_s": pt.pack_s,
        }
        if int4:
            out["int4_variant"] = int4
        if sweep:
            out["sweep"] = sweep
            out["sweep_note"] = ("per point: medians of 100 CUDA-event timings after 10 warm-ups; cold_l2 = "
                                 "256 MiB read before every run, warm_l2 = back to back; fwd = the layer call, "
                                 "k1/k2 = the kernels called one at a time; tflops, tokens_per_s, fractions "
                                 "and lowrank_overhead from the cold times")
        if not args.no_cpu_baseline:
            exp = layer.export()
            rc = exp["R_codes"]
            exp["R_codes"] = np.stack([rc & 0xF, rc >> 4], axis=-1).reshape(rc.shape[0], -1)
            v, rows, dt = oracle_sample(w, pt.d, exp)
            threads = blas_threads()
            out["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)),
                                   "threads": threads, "kind": "oracle",
                                   "sample": f"oracle forward on {rows} of {M} token rows ({dt:.2f} s) with the layer's packed operands"}
        print(json.dumps(out), flush=True)
    pt.close()
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------------ AWQ-style W4A16 layer
AWQ_METRIC = "AWQ-style W4A16 linear at the FLUX modulation shape: packed-weight GB/s and tokens/s"


def awq_bytes(w):
    """Algorithmic HBM bytes of one forward: codes, (scale, zero) pairs, 1/s, bias, X, Y."""
    return w.N * w.K / 2 + w.N * (w.K // 64) * 8 + w.K * 4 + w.N * 2 + w.M * w.K * 2 + w.M * w.N * 2


def run_awq(args, w):
    """The modulation layers' weight-only 4-bit linear (its own JSON line; replicas like the main
    layer under torchrun)."""
    import torch
    import torch.distributed as dist
    from w4a4_rank_corrected_e2m1_b300 import svdq

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    d = synthetic.make(w)
    layer = svdq.AwqLayer(d["W"], bias=d["bias"], Xcal=synthetic.make_x(w, 64, seed=7), device=local)
    stream = torch.cuda.current_stream()
    Xs = [torch.from_numpy(synthetic.make_x(w, w.M, seed=sd).view(np.int16)).cuda() for sd in batch_seeds(rank, 4)]
    Y = torch.empty((w.M, w.N), dtype=torch.bfloat16, device="cuda")
    flush = L2Flush(torch)
    for i in range(args.warmup):
        layer.forward(Xs[i % 4], Y, w.M, stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = Clocks(torch.cuda.current_device())
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush()
        ev[i][0].record(stream)
        layer.forward(Xs[i % 4], Y, w.M, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    layer.check_error()
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    (ms,) = max_over_ranks([ms], world, "cuda")
    if rank == 0:
        hbm, _, src = peaks()
        by = awq_bytes(w)
        gbs = job_rate(by, world, ms * 1e-3) / 1e9
        per_gpu = by / (ms * 1e-3) / 1e9
        out = {
            "metric": AWQ_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u4 weights (group 64, f32 scale, zero point) x bf16 acts; f16 products, f32 sums",
            "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "K": w.K, "N": w.N, "group": 64,
                       "l2": "flushed before every timed step (a 256 MiB read, outside the timed events)",
                       "parallelism": f"replicas x{world}"},
            "tokens_per_s": job_rate(w.M, world, ms * 1e-3),
            "roofline": {"bound": "hbm", "kernel": "awq_gemv", "achieved": per_gpu, "peak": hbm, "unit": "GB/s",
                         "frac": per_gpu / hbm, "traffic": ncu_traffic(w.name, "awq_gemv"),
                         "traffic_unit": "bytes per launch (ncu)", "algorithmic_bytes": by,
                         "peak_source": f"{src} copy bandwidth"},
            "gpu_launches": args.steps * ((w.M + 7) // 8), "clocks": clk,
        }
        print(json.dumps(out), flush=True)
    layer.close()
    if world > 1:
        dist.destroy_process_group()


def run_reference_awq(args, w):
    """The AWQ oracle's forward on the host cores (weights quantised once, without the scale
    search, which does not change the forward's cost)."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    from oracle import awq
    d = synthetic.make(w)
    p = awq.pack(d["W"], d["bias"])
    for _ in range(min(args.warmup, 1)):
        awq.forward(d["X"], p)
    steps = max(1, min(args.steps, 5))
    t0 = time.perf_counter()
    for _ in range(steps):
        awq.forward(d["X"], p)
    dt = (time.perf_counter() - t0) / steps
    val = awq_bytes(w) / dt / 1e9
    print(json.dumps({
        "impl": "reference", "metric": AWQ_METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "K": w.K, "N": w.N, "group": 64},
        "tokens_per_s": w.M / dt,
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": len(os.sched_getaffinity(0)), "threads": blas_threads(),
                         "kind": "oracle", "sample": f"oracle AWQ forward, {steps} steps of {w.M} rows"},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)


# ------------------------------------------------------------------ MLP pair (fused epilogue)
PAIR_METRIC = "FLUX MLP pair (3072 -> 12288 -> GELU -> 3072) forward with the fused epilogue: TFLOP/s"


def pair_flops(pw):
    up, dn = pw.up, pw.down
    return 2.0 * up.M * (up.N * up.K + dn.N * dn.K) + 2.0 * up.M * (up.rank * (up.K + up.N) + dn.rank * (dn.K + dn.N))


def run_pair(args, pw):
    """The MLP pair, fused and unfused (its own JSON line; one GPU)."""
    import torch
    from w4a4_rank_corrected_e2m1_b300 import svdq

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    if int(os.environ.get("RANK", "0")) != 0:
        return
    stream = torch.cuda.current_stream()
    clocks = Clocks(torch.cuda.current_device())
    out = measure_mlp_pair(torch, svdq, pw, stream, L2Flush(torch), reps=args.steps, warm=args.warmup)
    clk = clocks.stop()
    us = out["cold_l2"]["fused_us"]
    print(json.dumps({
        "metric": PAIR_METRIC, "value": pair_flops(pw) / (us * 1e-6) / 1e12, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us * 1e-3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4(e2m1,e4m3)+bf16, f32 accumulate", "data": "synthetic",
        "config": {"workload": pw.name, "M": pw.up.M, "K": pw.up.K, "N_up": pw.up.N, "N": pw.down.N,
                   "ranks": [pw.up.rank, pw.down.rank],
                   "l2": "flushed before every timed step (a 256 MiB read, outside the timed events)"},
        "tokens_per_s": pw.up.M / (us * 1e-6), "pair": out,
        "gpu_launches": 4 * args.steps, "clocks": clk}), flush=True)


def run_reference_pair(args, pw):
    """The oracle's MLP pair on the host cores, on a bounded sample of token rows."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    from oracle import svdquant as sq
    d = synthetic.make(pw.up)
    rows = 16
    up = sq.pack(d["W"], d["bias"], pw.up.rank, Xcal_bits=d["X"][:256])
    G = sq.f64_to_bf16(sq.gelu(sq.bf16_to_f64(sq.f64_to_bf16(sq.forward(d["X"][:256], up)))))
    wd = synthetic.make_weights(pw.down)
    down = sq.pack(wd["W"], wd["bias"], pw.down.rank, Xcal_bits=G)
    steps = max(1, min(args.steps, 3))
    t0 = time.perf_counter()
    for i in range(steps):
        sq.mlp_pair_forward(d["X"][rows * i: rows * (i + 1)], up, down)
    dt = (time.perf_counter() - t0) / steps
    val = pair_flops(pw) * rows / pw.up.M / dt / 1e12
    print(json.dumps({
        "impl": "reference", "metric": PAIR_METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": 0, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": pw.name, "M": pw.up.M, "K": pw.up.K, "N_up": pw.up.N, "N": pw.down.N},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)),
                         "threads": blas_threads(), "kind": "oracle",
                         "sample": f"oracle pair forward on {rows} token rows per step, {steps} steps"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)


def main():
    args = parse()
    if args.workload == synthetic.MLP_PAIR.name:
        (run_reference_pair if args.impl == "reference" else run_pair)(args, synthetic.MLP_PAIR)
        return
    w = synthetic.get(args.workload)
    if args.impl == "reference":
        if w in synthetic.AWQ_WORKLOADS:
            run_reference_awq(args, w)
        else:
            run_reference(args, w)
    elif w in synthetic.AWQ_WORKLOADS:
        run_awq(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
