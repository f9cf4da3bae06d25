"""Benchmark of the MXFP8 norm-quant + GEMM hot path on GB300.

One step = one pass of the whole path over one batch of M tokens:
  1. fused Gemma RMSNorm + MXFP8 quantisation of the residual x (M x 6144),
  2. per contraction K of the workload: MXFP8 quantisation of the activation
     A (M x K) and its GEMM against the pre-quantised weight W (6144 x K),
     bf16 out.
Weights are quantised once, before timing (serving loads MXFP8 weights).

The default workload is the largest single-GPU configuration, m32768_stress:
32768 tokens, the down_proj GEMM (K = 3072) and the 32768 x 6144 stress
residual (outlier channels, zero blocks, a zero row).  The same JSON line
carries a `sweep` record: every (M, K) point of the M sweep (M = 128 ...
32768, K = 2048 and 3072) and the m4096_rowscale workload, each kernel timed
alone (GEMM TFLOP/s and fraction of FP8 peak, norm-quant and quant GB/s and
fraction of HBM bandwidth).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload m32768_stress]
    python bench.py --impl reference ...   # the CPU oracle, timed on a bounded sample
    python bench.py --kernel gemm --workload sweep_m4096_k3072   # one kernel alone

Prints one JSON line (rank 0).  With N > 1 (torchrun) every rank runs the same
per-GPU workload on its own batch (weak scaling, no collective on the data
path); the barrier-bracketed time is the max over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

H = 6144
N_OUT = 6144
EPS = 1e-6
L2_BYTES = 129 * 1024 * 1024
FP8_PER_BF16 = 2.0        # dense FP8 / dense BF16 tensor rate (4.5 / 2.25 PFLOP/s nominal)
METRIC = "MXFP8 GEMM TFLOP/s (% FP8 peak) & norm-quant GB/s, M=128-32768, N=6144"
DEFAULT_WORKLOAD = "m32768_stress"
NEXT_M = (1024, 4096, 32768)       # sizes at which the sweep also times the forms beyond the main path


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ measured DRAM traffic

def gemm_traffic_per_launch(workload, k):
    """DRAM bytes (read + write) of one GEMM launch of the workload from the
    ncu capture committed under profiles/, or None when no capture of this
    workload exists or the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "k_gemm_mxf8_traffic.json")
    try:
        rec = json.load(open(path))
        h = hashlib.sha256()
        for f in rec["source_files"]:
            h.update(open(os.path.join(ROOT, f), "rb").read())
        if h.hexdigest() != rec["source_sha256"]:
            return None
        return int(rec["workloads"][workload]["dram_bytes_per_launch"][str(k)])
    except (OSError, KeyError, ValueError, TypeError):
        return None


# ------------------------------------------------------------------ traffic model

def norm_quant_bytes(m, h=H):
    """Algorithmic HBM bytes of one fused norm-quant launch: read x (2 B/elem),
    write codes (1 B/elem) and scales (padded F8_128x4 buffer), read w once."""
    c = h // 32
    scale = (-(-m // 128) * 128) * (-(-c // 4) * 4)
    return 2 * m * h + m * h + scale + 2 * h


def norm_rowmajor_bytes(m, h=H):
    """The norm with row-major scales: x read, codes and m * h/32 scale bytes written, w read."""
    return 2 * m * h + m * h + m * (h // 32) + 2 * h


def norm_bf16_bytes(m, h=H):
    """The norm alone in bf16: x read, y written (2 B/elem each), w read."""
    return 4 * m * h + 2 * h


def swizzle_bytes(m, h=H):
    """Row-major scales read, the padded F8_128x4 buffer written."""
    c = h // 32
    return m * c + (-(-m // 128) * 128) * (-(-c // 4) * 4)


def quant_bytes(r, c):
    cs = c // 32
    return 2 * r * c + r * c + (-(-r // 128) * 128) * (-(-cs // 4) * 4)


def gemm_flops(m, n, k):
    return 2.0 * m * n * k


def gemm_bytes(m, n, k):
    sa = (-(-m // 128) * 128) * (k // 32)
    sb = (-(-n // 128) * 128) * (k // 32)
    return m * k + sa + n * k + sb + 2 * m * n


def aggregate_over_ranks(ms_per_step, work_per_step, world, device=None):
    """Weak scaling: every rank did `work_per_step` per step; the job's step
    time is the slowest rank's.  Returns (max ms per step, whole-job work per
    second).  A rank-independent collective on the timing only; the data path
    has none."""
    import torch
    ms_max = float(ms_per_step)
    if world > 1:
        t = torch.tensor([ms_max], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms_max = float(t.item())
    return ms_max, world * work_per_step / (ms_max * 1e-3)


def make_config(wl, world):
    """The workload description both arms print (identical keys and values)."""
    return {"workload": wl.name, "M": wl.m, "N": N_OUT, "K": list(wl.ks), "norm_quant": f"{wl.norm_rows}x{H}",
            "step": "norm-quant(x) + per K: quant(A) + gemm(A, W pre-quantised)",
            "l2": "inputs larger than L2: rotating input and weight sets of more than 2x L2 between "
                  "consecutive launches of a buffer (no flush)",
            "parallelism": f"weak, {world} independent rank(s)"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            if t0 <= ts <= t1:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------ timing helpers

def graph_time(torch, stream, launch, n, replays):
    """Captures launch(0) ... launch(n-1) as one CUDA graph on `stream`,
    replays it once untimed, then `replays` times, each bracketed by CUDA
    events on the stream.  Returns the per-replay times in ms."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            launch(i)
    times = []
    with torch.cuda.stream(stream):
        g.replay()
        stream.synchronize()
        for _ in range(replays):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            stream.synchronize()
            times.append(e0.elapsed_time(e1))
    del g
    return times


def per_launch_stats(times_ms, n):
    """Median, min and max time of one launch in µs from per-replay times of n launches."""
    per = [t / n * 1e3 for t in times_ms]
    return statistics.median(per), min(per), max(per)


def rotation(bytes_per_launch):
    """Launches per timed replay: enough that one replay moves more than
    2.2x L2 through HBM, and at least 20."""
    return max(20, math.ceil(2.2 * L2_BYTES / max(1, bytes_per_launch)))


# ------------------------------------------------------------------ GPU arm

def run_gpu(args, rank, world):
    import torch

    import mxfp8_norm_quant_gb300 as mx
    from mxfp8_norm_quant_gb300 import workloads as W

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    mx.lib()
    wl = W.get_workload(args.workload)
    M = wl.m
    ks = wl.ks
    stream = torch.cuda.Stream(dev)
    sptr = stream.cuda_stream
    peaks = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_PER_BF16

    # ---- inputs, resident in HBM; R rotating sets so that the working set of
    # consecutive steps exceeds L2 (no flush needed between steps)
    x_h, w_h = wl.norm(seed=rank)
    a_h, wt_h = {}, {}
    for k in ks:
        a_h[k], wt_h[k] = wl.gemm(k, seed=rank)
    w_dev = w_h.to(dev)
    wq = {}
    for k in ks:
        wd = wt_h[k].to(dev)
        wq[k] = mx.quant(wd)
        del wd
    set_bytes = 2 * wl.norm_rows * H + wl.norm_rows * H + mx.mx_scale_bytes(wl.norm_rows, H)
    for k in ks:
        set_bytes += 3 * M * k + mx.mx_scale_bytes(M, k) + 2 * M * N_OUT
    weight_bytes = sum(N_OUT * k + mx.mx_scale_bytes(N_OUT, k) for k in ks)
    Mn = wl.norm_rows
    # each kernel alone must also cycle through more than 2.2x L2 of its own
    # inputs and outputs, so the sets are as many as the smallest kernel needs
    kernel_bytes = {"norm_quant": norm_quant_bytes(Mn)}
    for k in ks:
        kernel_bytes[f"quant_a{k}"] = quant_bytes(M, k)
        kernel_bytes[f"gemm_k{k}"] = gemm_bytes(M, N_OUT, k)
    alone_sets = {n: max(1, math.ceil(2.2 * L2_BYTES / b)) for n, b in kernel_bytes.items()}
    R = max(2, math.ceil(2.2 * L2_BYTES / max(1, set_bytes + weight_bytes)), max(alone_sets.values()))
    R = min(R, 160)
    sets = []
    for r in range(R):
        s = {"x": x_h.to(dev), "q": torch.empty((Mn, H), dtype=torch.uint8, device=dev),
             "s": torch.empty(mx.mx_scale_bytes(Mn, H), dtype=torch.uint8, device=dev)}
        for k in ks:
            s[f"a{k}"] = a_h[k].to(dev)
            s[f"aq{k}"] = torch.empty((M, k), dtype=torch.uint8, device=dev)
            s[f"as{k}"] = torch.empty(mx.mx_scale_bytes(M, k), dtype=torch.uint8, device=dev)
            s[f"c{k}"] = torch.empty((M, N_OUT), dtype=torch.bfloat16, device=dev)
        sets.append(s)
    # weights rotate too (each decoder layer has its own)
    wsets = [wq] + [{k: (wq[k][0].clone(), wq[k][1].clone()) for k in ks} for _ in range(R - 1)]
    torch.cuda.synchronize()

    def step(i):
        s = sets[i % R]
        wsx = wsets[i % R]
        mx.mx_rmsnorm_quant(s["x"], w_dev, EPS, s["q"], s["s"], Mn, H, sptr)
        for k in ks:
            mx.mx_quant_weights(s[f"a{k}"], s[f"aq{k}"], s[f"as{k}"], M, k, sptr)
            mx.mx_gemm(s[f"aq{k}"], s[f"as{k}"], wsx[k][0], wsx[k][1], s[f"c{k}"], M, N_OUT, k, sptr)

    def one_kernel(i, idx):
        s = sets[i % R]
        wsx = wsets[i % R]
        if idx == 0:
            mx.mx_rmsnorm_quant(s["x"], w_dev, EPS, s["q"], s["s"], Mn, H, sptr)
            return
        k = ks[(idx - 1) // 2]
        if (idx - 1) % 2 == 0:
            mx.mx_quant_weights(s[f"a{k}"], s[f"aq{k}"], s[f"as{k}"], M, k, sptr)
        else:
            mx.mx_gemm(s[f"aq{k}"], s[f"as{k}"], wsx[k][0], wsx[k][1], s[f"c{k}"], M, N_OUT, k, sptr)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    stream.synchronize()
    assert mx.mx_device_fault() == 0

    # The K timed steps are captured once as a CUDA graph (the launches go
    # through the same C entry points; the graph removes the host's per-call
    # launch latency, as a serving engine's CUDA-graph mode does).  The graph
    # is replayed `replays` times, each replay timed on its own; the step time
    # is the median replay / K.
    g_main = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_main, stream=stream):
        for i in range(args.steps):
            step(i)
    torch.cuda.synchronize()

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    # soak ~1.5 s so the clocks under load are sampled and settled
    t_soak = time.time()
    with torch.cuda.stream(stream):
        while time.time() - t_soak < 1.5:
            for _ in range(3):
                g_main.replay()
            stream.synchronize()

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    replay_ms = []
    with torch.cuda.stream(stream):
        for _ in range(args.replays):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g_main.replay()
            e1.record(stream)
            stream.synchronize()
            replay_ms.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_wall1 = time.time()
    clocks = sampler.summary(t_soak, t_wall1)
    ms_per_step = statistics.median(replay_ms) / args.steps

    order = ["norm_quant"]
    for k in ks:
        order += [f"quant_a{k}", f"gemm_k{k}"]
    # per-kernel durations inside the step: the same K steps captured again
    # with a CUDA event on the stream before and after every launch (event
    # nodes of the graph), replayed; a kernel's time is the sum over the K
    # steps of its events' interval, per launch, median over replays.  The
    # events end each kernel's overlap with the next one's set-up, so this
    # graph runs a little longer than the timed one.
    ev = [[(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
           for _ in order] for _ in range(args.steps)]
    g_inst = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_inst, stream=stream):
        for i in range(args.steps):
            for idx in range(len(order)):
                ev[i][idx][0].record(stream)
                one_kernel(i, idx)
                ev[i][idx][1].record(stream)
    n_inst = max(5, args.replays // 2)
    in_step = {name: [] for name in order}
    inst_ms = []
    with torch.cuda.stream(stream):
        for _ in range(n_inst):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g_inst.replay()
            e1.record(stream)
            stream.synchronize()
            inst_ms.append(e0.elapsed_time(e1))
            for idx, name in enumerate(order):
                in_step[name].append(sum(ev[i][idx][0].elapsed_time(ev[i][idx][1]) for i in range(args.steps)))
    del g_inst
    in_step_stats = {name: per_launch_stats(t, args.steps) for name, t in in_step.items()}
    # and each kernel alone: a graph of its K launches (same rotating
    # buffers), replayed and timed like the step
    alone = {}
    for idx, name in enumerate(order):
        n_al = max(args.steps, min(R, alone_sets[name]))
        t = graph_time(torch, stream, lambda i: one_kernel(i, idx), n_al, n_inst)
        alone[name] = per_launch_stats(t, n_al)
    sampler.stop()
    assert mx.mx_device_fault() == 0
    # The events cost time of their own (the graph's event nodes delay the
    # launch after them): the instrumented step minus the step, per launch.
    # A kernel whose time is not at least 20x that cost is reported alone.
    inst_ms_per_step = statistics.median(inst_ms) / args.steps
    event_cost_us = max(0.0, (inst_ms_per_step - ms_per_step) * 1e3 / len(order))
    per_kernel, timed_how = {}, {}
    for name in order:
        in_step_ok = event_cost_us <= 0.05 * in_step_stats[name][0]
        per_kernel[name] = in_step_stats[name] if in_step_ok else alone[name]
        timed_how[name] = "in the step" if in_step_ok else "alone"

    flops_step = sum(gemm_flops(M, N_OUT, k) for k in ks)
    kern = {}
    denom = sum(v[0] for v in per_kernel.values())
    for name in order:
        us, us_min, us_max = per_kernel[name]
        rec = {"us": us, "us_min": us_min, "us_max": us_max, "share": us / denom}
        if name == "norm_quant":
            b = norm_quant_bytes(Mn)
            rec.update({"GB/s": b / (us * 1e-6) / 1e9, "frac_hbm": b / (us * 1e-6) / 1e9 / peaks["hbm_gbs"]})
        elif name.startswith("quant_a"):
            b = quant_bytes(M, int(name[7:]))
            rec.update({"GB/s": b / (us * 1e-6) / 1e9, "frac_hbm": b / (us * 1e-6) / 1e9 / peaks["hbm_gbs"]})
        else:
            f = gemm_flops(M, N_OUT, int(name[6:]))
            rec.update({"TFLOP/s": f / (us * 1e-6) / 1e12, "frac_fp8": f / (us * 1e-6) / 1e12 / fp8_peak})
        rec["timed"] = timed_how[name]
        rec["in_step_us"] = in_step_stats[name][0]
        rec["alone_us"] = alone[name][0]
        kern[name] = rec
    plan = {k: mx.mx_gemm_plan(M, N_OUT, k) for k in ks}

    # the dominant kernel of the step and its roofline
    dom = max(order, key=lambda n: per_kernel[n][0])
    if dom.startswith("gemm_k"):
        # Timed inside the long run of the step (the clock record shows the
        # power cap active), the kernel's denominator is the sustained
        # measured peak; timed alone, the burst one.  The burst fraction is
        # reported beside it either way.
        k = int(dom[6:])
        in_step = timed_how[dom] == "in the step"
        fp8_sust = peaks["bf16_tflops_sustained"] * FP8_PER_BF16
        peak = fp8_sust if in_step else fp8_peak
        ach = kern[dom]["TFLOP/s"]
        how = ("sustained bf16 {} TFLOP/s x {} (nominal dense FP8/BF16 ratio), of measured: the kernel is timed "
               "inside the step's long run under the power cap").format(peaks["bf16_tflops_sustained"], FP8_PER_BF16)
        if not in_step:
            how = ("burst bf16 {} TFLOP/s x {} (nominal dense FP8/BF16 ratio), of measured: the kernel is timed "
                   "alone").format(peaks["bf16_tflops"], FP8_PER_BF16)
        roof = {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "traffic": gemm_traffic_per_launch(wl.name, k),
                "kernel": f"k_gemm_mxf8, {M}x{N_OUT}x{k}, one launch per step",
                "algorithmic": {"flops_per_launch": gemm_flops(M, N_OUT, k),
                                "bytes_per_launch": gemm_bytes(M, N_OUT, k)},
                "peak_source": f"{peaks['source']} {how}",
                "peak_burst": fp8_peak, "frac_of_burst": ach / fp8_peak}
    else:
        b = norm_quant_bytes(Mn) if dom == "norm_quant" else quant_bytes(M, int(dom[7:]))
        roof = {"bound": "hbm", "achieved": kern[dom]["GB/s"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": kern[dom]["frac_hbm"], "traffic": None, "kernel": dom,
                "algorithmic": {"bytes_per_launch": b}, "peak_source": f"{peaks['source']} HBM copy"}

    # ---- end to end through the C ABI with host buffers
    e2e = run_e2e(args, mx, torch, dev, stream, wl, x_h, w_dev, a_h, wq, ks)

    # ---- aggregate over ranks: max time, sum of work
    ms_max, value = aggregate_over_ranks(ms_per_step, flops_step / 1e12, world, dev)

    del sets, wsets, wq, g_main
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    sweep = None
    if not args.no_sweep:
        sweep = run_sweep(args, mx, torch, dev, stream, peaks, fp8_peak)
        assert mx.mx_device_fault() == 0

    nq = kern["norm_quant"]
    out = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3+ue8m0 in, fp32 accumulate, bf16 out",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights, U(-0.1,0.1) norm gain"
                + ("; residual with 61 x50 outlier channels, 1/128 zero blocks, row 0 zero)" if wl.stress else ")"),
        "config": make_config(wl, world),
        "gemm_plan": plan,
        "norm_quant_gbs": nq["GB/s"],
        "kernels": kern,
        "roofline": roof,
        "norm_quant_roofline": {"bound": "hbm", "achieved": nq["GB/s"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": nq["frac_hbm"], "peak_source": f"{peaks['source']} HBM copy"},
        "e2e": e2e,
        "gpu_launches": len(order) * args.steps * args.replays,
        "timing": {"timed_region": f"the K={args.steps}-step CUDA graph, replayed {args.replays} times, each "
                                   "replay timed with CUDA events on the launch stream",
                   "ms_per_step_median": ms_per_step,
                   "ms_per_step_min": min(replay_ms) / args.steps,
                   "ms_per_step_max": max(replay_ms) / args.steps,
                   "gpu_launches_per_replay": len(order) * args.steps,
                   "rotating_sets": R,
                   "rotating_MiB": round((set_bytes + weight_bytes) * R / 2**20),
                   "per_kernel": "in_step_us: inside the step, from CUDA events recorded before and after "
                                 "every launch of the K-step graph (a second capture of the same steps, replayed "
                                 f"{n_inst} times; median per launch); alone_us: a CUDA graph of max(K, enough "
                                 "for 2.2x L2 of the kernel's own bytes) launches over the rotating sets, "
                                 "replayed and timed the same way; us: the "
                                 "in-step time where the events' own cost per launch (instrumented step minus "
                                 "step) is at most 5 % of it, else the time alone (`timed` says which)",
                   "instrumented_ms_per_step": inst_ms_per_step,
                   "event_cost_us_per_launch": event_cost_us},
        "clocks": clocks,
        "wall_s_timed": t_wall1 - t_wall0,
    }
    if sweep is not None:
        out["sweep"] = sweep
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        out["cpu_baseline"] = cpu_baseline(wl, ks)
    return out


def run_sweep(args, mx, torch, dev, stream, peaks, fp8_peak):
    """Each kernel of the path timed alone at every point of the M sweep
    (M = 128 ... 32768, K = 2048 and 3072, N = H = 6144) and on the
    m4096_rowscale workload.  Inputs: the seeded 32768-row sweep tensors (the
    first M rows are exactly the sweep_m<M> workload), held twice over in
    one device pool; the launches of one timed replay cycle over row windows
    of the pool (and over copies of the weight) so that every replay moves
    more than 2.2x L2 through HBM."""
    from mxfp8_norm_quant_gb300 import workloads as W
    sptr = stream.cuda_stream
    reps = args.sweep_replays
    Mmax = max(W.M_SWEEP)
    pool = 2 * Mmax
    cp = (H // 32 + 3) // 4 * 4                      # scale bytes per row of a 6144-wide operand
    pts = {}

    def windows(m):
        return pool // m                             # row windows of the pool at offsets j*m (j*m % 128 == 0)

    # ---- norm-quant
    x_h, w_h = W.norm_inputs(Mmax, H, seed=0)
    x_pool = torch.empty((pool, H), dtype=torch.bfloat16, device=dev)
    x_pool[:Mmax].copy_(x_h.to(dev))
    x_pool[Mmax:].copy_(x_pool[:Mmax])
    del x_h
    q_pool = torch.empty((pool, H), dtype=torch.uint8, device=dev)
    s_pool = torch.empty(pool * cp, dtype=torch.uint8, device=dev)
    w_dev = w_h.to(dev)
    norm_pts = []
    for m in W.M_SWEEP:
        nw = windows(m)
        n = rotation(norm_quant_bytes(m))

        def launch(i, m=m, nw=nw):
            r0 = (i % nw) * m
            mx.mx_rmsnorm_quant(x_pool[r0:r0 + m], w_dev, EPS, q_pool[r0:r0 + m], s_pool[r0 * cp:(r0 + m) * cp],
                                m, H, sptr)
        us, lo, hi = per_launch_stats(graph_time(torch, stream, launch, n, reps), n)
        gbs = norm_quant_bytes(m) / (us * 1e-6) / 1e9
        norm_pts.append({"M": m, "us": us, "us_min": lo, "us_max": hi, "GB/s": gbs,
                         "frac_hbm": gbs / peaks["hbm_gbs"], "launches_per_replay": n})
    # ---- the sequence-parallel forms of the norm (row-major scales, BF16 y)
    # and the standalone swizzle, on the same pool
    next_pts = []
    y_pool = torch.empty((pool, H), dtype=torch.bfloat16, device=dev)
    sw_pool = torch.empty(pool * cp, dtype=torch.uint8, device=dev)
    for m in NEXT_M:
        nw = windows(m)

        def lr(i, m=m, nw=nw):
            r0 = (i % nw) * m
            mx.mx_rmsnorm_quant_ex(x_pool[r0:r0 + m], w_dev, EPS, q_pool[r0:r0 + m], s_pool[r0 * 192:(r0 + m) * 192],
                                   m, H, mx.MX_SCALES_ROW_MAJOR, sptr)

        def lb(i, m=m, nw=nw):
            r0 = (i % nw) * m
            mx.mx_rmsnorm_bf16(x_pool[r0:r0 + m], w_dev, EPS, y_pool[r0:r0 + m], m, H, sptr)

        def ls(i, m=m, nw=nw):
            r0 = (i % nw) * m
            mx.mx_swizzle_scales(s_pool[r0 * 192:(r0 + m) * 192], sw_pool[r0 * cp:(r0 + m) * cp], m, H, sptr)
        for name, fn, nbytes in (("norm_rowmajor", lr, norm_rowmajor_bytes(m)), ("norm_bf16", lb, norm_bf16_bytes(m)),
                                 ("swizzle", ls, swizzle_bytes(m))):
            n = rotation(nbytes)
            us, lo, hi = per_launch_stats(graph_time(torch, stream, fn, n, reps), n)
            gbs = nbytes / (us * 1e-6) / 1e9
            next_pts.append({"kernel": name, "M": m, "us": us, "us_min": lo, "us_max": hi, "GB/s": gbs,
                             "frac_hbm": gbs / peaks["hbm_gbs"]})
    del x_pool, q_pool, s_pool, y_pool, sw_pool
    torch.cuda.empty_cache()

    # ---- quant + GEMM per K
    gemm_pts = []
    for k in (W.K_OPROJ, W.K_DOWN):
        a_h, wt_h = W.gemm_operands(Mmax, k, seed=0)
        a_pool = torch.empty((pool, k), dtype=torch.bfloat16, device=dev)
        a_pool[:Mmax].copy_(a_h.to(dev))
        a_pool[Mmax:].copy_(a_pool[:Mmax])
        del a_h
        cpk = (k // 32 + 3) // 4 * 4
        aq_pool = torch.empty((pool, k), dtype=torch.uint8, device=dev)
        as_pool = torch.empty(pool * cpk, dtype=torch.uint8, device=dev)
        mx.mx_quant_weights(a_pool, aq_pool, as_pool, pool, k, sptr)
        wq0 = mx.quant(wt_h.to(dev), stream=sptr)
        wbytes = N_OUT * k + mx.mx_scale_bytes(N_OUT, k)
        nwq = max(3, min(24, math.ceil(2.2 * L2_BYTES / wbytes)))
        wqs = [wq0] + [(wq0[0].clone(), wq0[1].clone()) for _ in range(nwq - 1)]
        c_pool = torch.empty((pool, N_OUT), dtype=torch.bfloat16, device=dev)
        cq_pool = torch.empty((pool, N_OUT), dtype=torch.uint8, device=dev)
        cs_pool = torch.empty(pool * cp, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        for m in W.M_SWEEP:
            nw = windows(m)
            ng = rotation(gemm_bytes(m, N_OUT, k))

            def lg(i, m=m, nw=nw):
                r0 = (i % nw) * m
                wq_ = wqs[i % nwq]
                mx.mx_gemm(aq_pool[r0:r0 + m], as_pool[r0 * cpk:(r0 + m) * cpk], wq_[0], wq_[1],
                           c_pool[r0:r0 + m], m, N_OUT, k, sptr)
            us, lo, hi = per_launch_stats(graph_time(torch, stream, lg, ng, reps), ng)
            tf = gemm_flops(m, N_OUT, k) / (us * 1e-6) / 1e12
            nq_ = rotation(quant_bytes(m, k))

            def lq(i, m=m, nw=nw):
                r0 = (i % nw) * m
                mx.mx_quant_weights(a_pool[r0:r0 + m], aq_pool[r0:r0 + m], as_pool[r0 * cpk:(r0 + m) * cpk],
                                    m, k, sptr)
            qus, qlo, qhi = per_launch_stats(graph_time(torch, stream, lq, nq_, reps), nq_)
            qgbs = quant_bytes(m, k) / (qus * 1e-6) / 1e9
            plan = mx.mx_gemm_plan(m, N_OUT, k)
            gemm_pts.append({"M": m, "K": k, "gemm_us": us, "gemm_us_min": lo, "gemm_us_max": hi,
                             "gemm_tflops": tf, "frac_fp8": tf / fp8_peak,
                             "tile": [plan["tile_m"], plan["tile_n"]],
                             "quant_us": qus, "quant_gbs": qgbs, "quant_frac_hbm": qgbs / peaks["hbm_gbs"]})
            if m in NEXT_M:
                # the GEMM whose epilogue emits C as MXFP8 (codes + F8_128x4 scales)
                def lgq(i, m=m, nw=nw):
                    r0 = (i % nw) * m
                    wq_ = wqs[i % nwq]
                    mx.mx_gemm_quant(aq_pool[r0:r0 + m], as_pool[r0 * cpk:(r0 + m) * cpk], wq_[0], wq_[1],
                                     cq_pool[r0:r0 + m], cs_pool[r0 * cp:(r0 + m) * cp], m, N_OUT, k, 0, 0, sptr)
                n = rotation(gemm_bytes(m, N_OUT, k))
                gus, glo, ghi = per_launch_stats(graph_time(torch, stream, lgq, n, reps), n)
                gtf = gemm_flops(m, N_OUT, k) / (gus * 1e-6) / 1e12
                next_pts.append({"kernel": "gemm_quant", "M": m, "K": k, "us": gus, "us_min": glo, "us_max": ghi,
                                 "TFLOP/s": gtf, "frac_fp8": gtf / fp8_peak})
        del a_pool, aq_pool, as_pool, wqs, wq0, c_pool, cq_pool, cs_pool
        torch.cuda.empty_cache()

    # ---- m4096_rowscale: LogUniform row scales on A and x
    wl = W.WORKLOADS["m4096_rowscale"]
    m = wl.m
    rs = {}
    xr, wr = wl.norm(seed=0)
    nsets = max(3, math.ceil(2.2 * L2_BYTES / norm_quant_bytes(m)))
    xs = [xr.to(dev) for _ in range(nsets)]
    wrd = wr.to(dev)
    qs = [torch.empty((m, H), dtype=torch.uint8, device=dev) for _ in range(nsets)]
    ss = [torch.empty(mx.mx_scale_bytes(m, H), dtype=torch.uint8, device=dev) for _ in range(nsets)]

    def ln(i):
        j = i % nsets
        mx.mx_rmsnorm_quant(xs[j], wrd, EPS, qs[j], ss[j], m, H, sptr)
    n = rotation(norm_quant_bytes(m))
    us, lo, hi = per_launch_stats(graph_time(torch, stream, ln, n, reps), n)
    gbs = norm_quant_bytes(m) / (us * 1e-6) / 1e9
    rs["norm_quant"] = {"M": m, "us": us, "us_min": lo, "us_max": hi, "GB/s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"]}
    del xs, qs, ss
    for k in wl.ks:
        a, wt = wl.gemm(k, seed=0)
        per = gemm_bytes(m, N_OUT, k)
        nsets = max(3, math.ceil(2.2 * L2_BYTES / per))
        ad = [a.to(dev) for _ in range(nsets)]
        ops = [mx.quant(t, stream=sptr) for t in ad]
        wqs = [mx.quant(wt.to(dev), stream=sptr) for _ in range(nsets)]
        cs = [torch.empty((m, N_OUT), dtype=torch.bfloat16, device=dev) for _ in range(nsets)]

        def lg(i, k=k):
            j = i % nsets
            mx.mx_gemm(ops[j][0], ops[j][1], wqs[j][0], wqs[j][1], cs[j], m, N_OUT, k, sptr)

        def lq(i, k=k):
            j = i % nsets
            mx.mx_quant_weights(ad[j], ops[j][0], ops[j][1], m, k, sptr)
        n = rotation(per)
        us, lo, hi = per_launch_stats(graph_time(torch, stream, lg, n, reps), n)
        tf = gemm_flops(m, N_OUT, k) / (us * 1e-6) / 1e12
        n = rotation(quant_bytes(m, k))
        qus, _, _ = per_launch_stats(graph_time(torch, stream, lq, n, reps), n)
        qgbs = quant_bytes(m, k) / (qus * 1e-6) / 1e9
        rs[f"k{k}"] = {"gemm_us": us, "gemm_us_min": lo, "gemm_us_max": hi, "gemm_tflops": tf,
                       "frac_fp8": tf / fp8_peak, "quant_us": qus, "quant_gbs": qgbs,
                       "quant_frac_hbm": qgbs / peaks["hbm_gbs"]}
        del ad, ops, wqs, cs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return {"note": "each kernel alone: a CUDA graph of >= 20 launches cycling over row windows of a "
                    "device pool holding the seeded 32768-row sweep tensors twice (the first M rows are the "
                    f"sweep_m<M> workload) and over weight copies, > 2.2x L2 per replay; {reps} timed replays, "
                    "us = median per launch (min, max over replays)",
            "peaks": {"fp8_tflops": fp8_peak, "hbm_gbs": peaks["hbm_gbs"],
                      "source": f"{peaks['source']}; FP8 = bf16 x {FP8_PER_BF16}"},
            "gemm_quant": gemm_pts, "norm_quant": norm_pts, "m4096_rowscale": rs,
            "next": {"note": "the rows beyond the main path: the MXFP8-output GEMM (automatic tile), the norm with "
                             "row-major scales and in BF16, and the standalone F8_128x4 swizzle of row-major scales",
                     "points": next_pts}}


def run_e2e(args, mx, torch, dev, stream, wl, x_h, w_dev, a_h, wq, ks):
    """Same metric end to end: every step copies its inputs from pinned host
    memory to the device, runs the step through the C ABI and copies all of
    its outputs (codes, scales, C) back to pinned host memory.  Steps are
    pipelined as a serving loop runs them: copy-in, compute and copy-out on
    three streams with double-buffered device and host buffers, so step i's
    compute overlaps step i+1's copy-in and step i-1's copy-out.  The timed
    region runs from before the first copy-in to after the last copy-out."""
    M = wl.m
    Mn = wl.norm_rows
    x_pin = x_h.pin_memory()
    a_pin = {k: a_h[k].pin_memory() for k in ks}

    def buffers():
        b = {"x": torch.empty_like(x_pin, device=dev),
             "q": torch.empty((Mn, H), dtype=torch.uint8, device=dev),
             "s": torch.empty(mx.mx_scale_bytes(Mn, H), dtype=torch.uint8, device=dev)}
        for k in ks:
            b[f"a{k}"] = torch.empty_like(a_pin[k], device=dev)
            b[f"aq{k}"] = torch.empty((M, k), dtype=torch.uint8, device=dev)
            b[f"as{k}"] = torch.empty(mx.mx_scale_bytes(M, k), dtype=torch.uint8, device=dev)
            b[f"c{k}"] = torch.empty((M, N_OUT), dtype=torch.bfloat16, device=dev)
        b["q_h"] = torch.empty_like(b["q"], device="cpu").pin_memory()
        b["s_h"] = torch.empty_like(b["s"], device="cpu").pin_memory()
        for k in ks:
            b[f"c{k}_h"] = torch.empty_like(b[f"c{k}"], device="cpu").pin_memory()
        return b

    bufs = [buffers(), buffers()]
    h2d = x_pin.numel() * 2 + sum(a_pin[k].numel() * 2 for k in ks)
    d2h = bufs[0]["q"].numel() + bufs[0]["s"].numel() + sum(bufs[0][f"c{k}"].numel() * 2 for k in ks)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_comp = stream
    ev = lambda: torch.cuda.Event()
    in_done = [ev(), ev()]
    comp_done = [ev(), ev()]
    out_done = [ev(), ev()]
    for e in in_done + comp_done + out_done:
        e.record(s_comp)

    def step(i):
        b = bufs[i % 2]
        j = i % 2
        # copy-in: buffer j's inputs were last read by the compute of step i-2
        s_in.wait_event(comp_done[j])
        with torch.cuda.stream(s_in):
            b["x"].copy_(x_pin, non_blocking=True)
            for k in ks:
                b[f"a{k}"].copy_(a_pin[k], non_blocking=True)
        in_done[j].record(s_in)
        # compute: its outputs were last read by the copy-out of step i-2
        s_comp.wait_event(in_done[j])
        s_comp.wait_event(out_done[j])
        sp = s_comp.cuda_stream
        mx.mx_rmsnorm_quant(b["x"], w_dev, EPS, b["q"], b["s"], Mn, H, sp)
        for k in ks:
            mx.mx_quant_weights(b[f"a{k}"], b[f"aq{k}"], b[f"as{k}"], M, k, sp)
            mx.mx_gemm(b[f"aq{k}"], b[f"as{k}"], wq[k][0], wq[k][1], b[f"c{k}"], M, N_OUT, k, sp)
        comp_done[j].record(s_comp)
        # copy-out
        s_out.wait_event(comp_done[j])
        with torch.cuda.stream(s_out):
            b["q_h"].copy_(b["q"], non_blocking=True)
            b["s_h"].copy_(b["s"], non_blocking=True)
            for k in ks:
                b[f"c{k}_h"].copy_(b[f"c{k}"], non_blocking=True)
        out_done[j].record(s_out)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(args.steps):
        step(i)
    s_out.wait_event(comp_done[(args.steps - 1) % 2])
    s_out.wait_event(out_done[(args.steps - 1) % 2])
    e1.record(s_out)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    flops = sum(gemm_flops(M, N_OUT, k) for k in ks)
    # the host link on this machine, with the step's own copies and no compute:
    # the inputs in on one stream and the outputs out on another, at once;
    # the best of three trials of at least five copies and 2 GB each
    b = bufs[0]

    def copies():
        with torch.cuda.stream(s_in):
            b["x"].copy_(x_pin, non_blocking=True)
            for k in ks:
                b[f"a{k}"].copy_(a_pin[k], non_blocking=True)
        with torch.cuda.stream(s_out):
            b["q_h"].copy_(b["q"], non_blocking=True)
            b["s_h"].copy_(b["s"], non_blocking=True)
            for k in ks:
                b[f"c{k}_h"].copy_(b[f"c{k}"], non_blocking=True)

    trials = []
    n_copies = max(5, math.ceil(2e9 / (h2d + d2h)))
    for _ in range(3):
        torch.cuda.synchronize()
        l0 = torch.cuda.Event(enable_timing=True)
        l1 = torch.cuda.Event(enable_timing=True)
        l0.record(s_in)
        s_out.wait_event(l0)
        for _ in range(n_copies):
            copies()
        s_out.wait_stream(s_in)
        l1.record(s_out)
        torch.cuda.synchronize()
        trials.append(n_copies * (h2d + d2h) / (l0.elapsed_time(l1) * 1e-3) / 1e9)
    link_gbs = max(trials)
    step_gbs = (h2d + d2h) / (ms * 1e-3) / 1e9
    del bufs
    return {"value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipeline": "copy-in, compute and copy-out streams, double-buffered device and pinned host buffers",
            "host_link": {"copies_only_gbs": link_gbs, "trials_gbs": trials, "step_gbs": step_gbs,
                          "frac": step_gbs / link_gbs,
                          "what": "the step's own copies (inputs in, outputs out, on two streams at once) "
                                  "without compute, on this box, best of 3 trials of max(5, 2 GB) copies; a frac "
                                  "above 1 means the "
                                  "link was slower during these trials than during the timed steps (the host "
                                  "is shared)"}}


# ------------------------------------------------------------------ CPU oracle arm

def _blas_threads():
    """(threads numpy's BLAS runs the oracle GEMM on, how that was found)."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n), "threadpoolctl"
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var, "")
        if v.isdigit() and int(v) > 0:
            return int(v), var
    return os.cpu_count() or 1, "BLAS default: all host cores (no thread limit set)"


def _bits(t):
    import numpy as np
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def cpu_baseline(wl, ks, sample_rows=(256, 1024), chunk=4096):
    """The oracle as it stands, on the host cores, on the headline workload:
    the norm-quant over all of x (in row chunks, so the temporaries stay a
    few GB), and quant + GEMM of the first r rows of each A against the full
    weight for the two sample sizes r in `sample_rows`.  The quant + GEMM
    time is extrapolated to all M rows by the straight line through the two
    samples (a fixed part -- the GEMM decodes the whole weight each call --
    plus a per-row part); the extrapolation is labelled as such.  The norm
    and the quantiser run in numpy on one thread; the GEMM's float64 matmul
    uses the BLAS threads."""
    import oracle as O
    x, w = wl.norm(seed=0)
    xb, wb = _bits(x), _bits(w)
    Mn = xb.shape[0]
    t0 = time.time()
    for r in range(0, Mn, chunk):
        O.rmsnorm_quant(xb[r:r + chunk], wb, wl.eps)
    t_norm = time.time() - t0
    per_k = {}
    t_full = t_norm
    r1, r2 = sample_rows
    for k in ks:
        a, wt = wl.gemm(k, seed=0)
        bq, bs = O.quant(_bits(wt))                       # untimed: weights are pre-quantised
        ts = []
        for r in (r1, r2):
            ab = _bits(a[:r])
            t0 = time.time()
            aq, as_ = O.quant(ab)
            O.gemm_ref(aq, as_, bq, bs)
            ts.append(time.time() - t0)
        per_row = max(0.0, (ts[1] - ts[0]) / (r2 - r1))
        fixed = max(0.0, ts[0] - per_row * r1)
        full = fixed + per_row * wl.m
        t_full += full
        per_k[f"k{k}"] = {"sample_s": {str(r1): ts[0], str(r2): ts[1]},
                          "rows_per_s_marginal": (1.0 / per_row) if per_row > 0 else None,
                          "fixed_s": fixed, "quant_gemm_s_full_extrapolated": full,
                          "gemm_gflops_at_sample": gemm_flops(r2, N_OUT, k) / ts[1] / 1e9}
    flops = sum(gemm_flops(wl.m, N_OUT, k) for k in ks)
    blas, how = _blas_threads()
    return {"value": flops / t_full / 1e12, "unit": "TFLOP/s", "cores": blas,
            "kind": "oracle",
            "sample": f"norm-quant of all {Mn}x{H} rows measured ({t_norm:.1f} s); quant + GEMM measured on the "
                      f"first {r1} and {r2} of {wl.m} rows and extrapolated linearly to {wl.m} rows; value = GEMM "
                      "flops of one step / (measured norm-quant + extrapolated quant + GEMM time)",
            "norm_quant_full_s": t_norm,
            "norm_quant_gbs": norm_quant_bytes(Mn) / t_norm / 1e9,
            "per_k": per_k,
            "step_s_extrapolated": t_full,
            "threads": {"norm_quant": 1, "quant": 1, "gemm_blas": blas, "gemm_blas_source": how},
            "host_cpus": os.cpu_count()}


def _oracle_prepare(wl, ks, rows):
    """Untimed: seeded inputs as the oracle takes them, weights quantised by the oracle."""
    import oracle as O
    x, w = wl.norm(seed=0)
    ops = []
    for k in ks:
        a, wt = wl.gemm(k, seed=0)
        bq, bs = O.quant(_bits(wt))
        ops.append((k, _bits(a[:rows]), bq, bs))
    return {"x": _bits(x[:rows]), "w": _bits(w), "ops": ops, "rows": rows, "eps": wl.eps}


def _oracle_step(prep):
    """One bounded sample of a step, run by the oracle as it stands: norm-quant
    of `rows` rows of x, quantisation of `rows` rows of each A, and their GEMM
    rows against the full 6144-row weight.  Returns the GEMM flops done."""
    import oracle as O
    O.rmsnorm_quant(prep["x"], prep["w"], prep["eps"])
    flops = 0.0
    for k, ab, bq, bs in prep["ops"]:
        aq, as_ = O.quant(ab)
        O.gemm_ref(aq, as_, bq, bs)
        flops += gemm_flops(prep["rows"], N_OUT, k)
    return flops


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, each step one bounded sample of the workload."""
    from mxfp8_norm_quant_gb300 import workloads as W
    wl = W.get_workload(args.workload)
    ks = wl.ks
    rows = 64
    prep = _oracle_prepare(wl, ks, rows)
    for _ in range(args.warmup):
        _oracle_step(prep)
    t0 = time.time()
    flops = 0.0
    for _ in range(args.steps):
        flops += _oracle_step(prep)
    dt = time.time() - t0
    value = flops / dt / 1e12
    blas, how = _blas_threads()
    sample = (f"{args.steps} x ({rows} rows of norm-quant {wl.norm_rows}x{H}; {rows} rows of quant + GEMM vs the "
              f"full 6144-row weight for K={list(ks)}), {dt:.1f} s")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 GEMM of decoded MXFP8, f32 norm", "data": "synthetic",
        "config": make_config(wl, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas, "kind": "oracle", "sample": sample,
                         "threads": {"norm_quant": 1, "quant": 1, "gemm_blas": blas, "gemm_blas_source": how}},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_one_kernel(args):
    """--kernel mode: one kernel of the path, launched eagerly `steps` times on
    rotating buffers after `warmup` launches (used for ncu captures and sweeps).
    Reports the mean device time per launch from CUDA events."""
    import torch

    import mxfp8_norm_quant_gb300 as mx
    from mxfp8_norm_quant_gb300 import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = W.get_workload(args.workload)
    M = wl.m
    k = args.k if args.k else wl.ks[-1]
    stream = torch.cuda.Stream(dev)
    sptr = stream.cuda_stream
    # rotate over enough copies that the launches' inputs and outputs together
    # exceed L2 twice over, so every launch reads its inputs from HBM
    c_m = -(-M // 128) * 128
    set_bytes = {
        "norm_quant": 3 * M * H + c_m * H // 32, "norm_rowmajor": 3 * M * H + M * H // 32, "norm_bf16": 4 * M * H,
        "swizzle": 2 * c_m * H // 32, "quant": 3 * M * k + c_m * k // 32,
        "gemm": M * k + N_OUT * k + 2 * M * N_OUT, "gemm_quant": M * k + N_OUT * k + M * N_OUT,
    }[args.kernel]
    R = max(3, min(512, math.ceil(2.2 * L2_BYTES / set_bytes)))
    if args.kernel == "norm_quant":
        x, w = wl.norm()
        xs = [x.to(dev) for _ in range(R)]
        wd = w.to(dev)
        qs = [torch.empty((M, H), dtype=torch.uint8, device=dev) for _ in range(R)]
        ss = [torch.empty(mx.mx_scale_bytes(M, H), dtype=torch.uint8, device=dev) for _ in range(R)]

        def launch(i):
            mx.mx_rmsnorm_quant(xs[i % R], wd, EPS, qs[i % R], ss[i % R], M, H, sptr)
        work, unit = norm_quant_bytes(M) / 1e9, "GB/s"
    elif args.kernel in ("norm_rowmajor", "norm_bf16"):
        x, w = wl.norm()
        xs = [x.to(dev) for _ in range(R)]
        wd = w.to(dev)
        if args.kernel == "norm_bf16":
            ys = [torch.empty((M, H), dtype=torch.bfloat16, device=dev) for _ in range(R)]

            def launch(i):
                mx.mx_rmsnorm_bf16(xs[i % R], wd, EPS, ys[i % R], M, H, sptr)
            work = norm_bf16_bytes(M) / 1e9
        else:
            qs = [torch.empty((M, H), dtype=torch.uint8, device=dev) for _ in range(R)]
            ss = [torch.empty((M, H // 32), dtype=torch.uint8, device=dev) for _ in range(R)]

            def launch(i):
                mx.mx_rmsnorm_quant_ex(xs[i % R], wd, EPS, qs[i % R], ss[i % R], M, H, mx.MX_SCALES_ROW_MAJOR,
                                       sptr)
            work = norm_rowmajor_bytes(M) / 1e9
        unit = "GB/s"
    elif args.kernel == "swizzle":
        x, w = wl.norm()
        _, s_rm = mx.rmsnorm_quant_rowmajor(x.to(dev), w.to(dev), EPS)
        ins = [s_rm.clone() for _ in range(R)]
        outs = [torch.empty(mx.mx_scale_bytes(M, H), dtype=torch.uint8, device=dev) for _ in range(R)]

        def launch(i):
            mx.mx_swizzle_scales(ins[i % R], outs[i % R], M, H, sptr)
        work, unit = swizzle_bytes(M) / 1e9, "GB/s"
    elif args.kernel == "quant":
        a, _ = wl.gemm(k)
        xs = [a.to(dev) for _ in range(R)]
        qs = [torch.empty((M, k), dtype=torch.uint8, device=dev) for _ in range(R)]
        ss = [torch.empty(mx.mx_scale_bytes(M, k), dtype=torch.uint8, device=dev) for _ in range(R)]

        def launch(i):
            mx.mx_quant_weights(xs[i % R], qs[i % R], ss[i % R], M, k, sptr)
        work, unit = quant_bytes(M, k) / 1e9, "GB/s"
    elif args.kernel == "gemm_quant":
        a, wt = wl.gemm(k)
        ops = [mx.quant(a.to(dev)) for _ in range(R)]
        wqs = [mx.quant(wt.to(dev)) for _ in range(R)]
        qouts = [torch.empty((M, N_OUT), dtype=torch.uint8, device=dev) for _ in range(R)]
        souts = [torch.empty(mx.mx_scale_bytes(M, N_OUT), dtype=torch.uint8, device=dev) for _ in range(R)]

        def launch(i):
            j = i % R
            mx.mx_gemm_quant(ops[j][0], ops[j][1], wqs[j][0], wqs[j][1], qouts[j], souts[j], M, N_OUT, k,
                             args.tile_m, args.tile_n, sptr)
        work, unit = gemm_flops(M, N_OUT, k) / 1e12, "TFLOP/s"
    elif args.kernel == "gemm":
        a, wt = wl.gemm(k)
        ops = [mx.quant(a.to(dev)) for _ in range(R)]
        wqs = [mx.quant(wt.to(dev)) for _ in range(R)]
        outs = [torch.empty((M, N_OUT), dtype=torch.bfloat16, device=dev) for _ in range(R)]

        def launch(i):
            j = i % R
            mx.mx_gemm_ex(ops[j][0], ops[j][1], wqs[j][0], wqs[j][1], outs[j], M, N_OUT, k, args.tile_m,
                          args.tile_n, sptr)
        work, unit = gemm_flops(M, N_OUT, k) / 1e12, "TFLOP/s"
    else:
        raise SystemExit(f"unknown --kernel {args.kernel}")
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            launch(i)
        stream.synchronize()
        # every timed pass runs through all R sets at least once
        n = max(args.steps, R)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for i in range(n):
            evs[i][0].record(stream)
            launch(i)
            evs[i][1].record(stream)
        stream.synchronize()
        # the same launches captured in a CUDA graph: device time without the
        # host's launch latency between them
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                launch(i)
        g.replay()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        g.replay()
        g1.record(stream)
        stream.synchronize()
    assert mx.mx_device_fault() == 0
    ms = [a.elapsed_time(b) for a, b in evs]
    med = statistics.median(ms)
    g_us = g0.elapsed_time(g1) / n * 1e3
    out = {"kernel": args.kernel, "workload": wl.name, "M": M, "K": k if args.kernel in ("quant", "gemm", "gemm_quant") else None,
           "rotating_sets": R,
           "launches": n, "us_median": med * 1e3, "us_min": min(ms) * 1e3,
           "rate_median": work / (med * 1e-3), "rate_best": work / (min(ms) * 1e-3),
           "us_graph": g_us, "rate_graph": work / (g_us * 1e-6), "unit": unit}
    if args.kernel in ("gemm", "gemm_quant"):
        out["plan"] = mx.mx_gemm_plan(M, N_OUT, k)
        out["tile"] = [args.tile_m, args.tile_n] if args.tile_m else [out["plan"]["tile_m"], out["plan"]["tile_n"]]
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--replays", type=int, default=20, help="timed replays of the K-step graph (median reported)")
    ap.add_argument("--sweep-replays", type=int, default=7, help="timed replays per sweep point")
    ap.add_argument("--no-sweep", action="store_true", help="skip the per-config sweep record")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel", choices=["norm_quant", "norm_rowmajor", "norm_bf16", "swizzle", "quant", "gemm",
                                             "gemm_quant"],
                    help="time one kernel of the path alone (eager launches)")
    ap.add_argument("--k", type=int, default=0, help="--kernel mode: contraction size (default: workload's last)")
    ap.add_argument("--tile-m", type=int, default=0, help="--kernel gemm: force the tile (128 or 256 = CTA pair)")
    ap.add_argument("--tile-n", type=int, default=0, help="--kernel gemm: force the tile width")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    args.replays = max(1, args.replays)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.kernel:
        run_one_kernel(args)
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    out = run_gpu(args, rank, world)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
