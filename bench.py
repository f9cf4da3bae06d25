"""Benchmark of the MXFP8 norm-quant + GEMM hot path on GB300.

One step = one pass of the whole path over one batch of M tokens:
  1. fused Gemma RMSNorm + MXFP8 quantisation of the residual x (M x 6144),
  2. MXFP8 quantisation of the o_proj activation A (M x 2048) and its GEMM
     against the pre-quantised weight W (6144 x 2048), bf16 out,
  3. the same for the down_proj activation (M x 3072) and W (6144 x 3072).
Weights are quantised once, before timing (serving loads MXFP8 weights).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload m1024]
    python bench.py --impl reference ...   # the CPU oracle, timed on a bounded sample

Prints one JSON line (rank 0).  With N > 1 (torchrun) every rank runs the same
per-GPU workload on its own batch (weak scaling, no collective on the data
path); the barrier-bracketed time is the max over ranks.
"""

from __future__ import annotations

import argparse
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

def gemm_traffic_per_step(workload):
    """DRAM bytes (read + write) of the step's GEMM launches from the ncu
    capture committed under profiles/, or None when that capture is of
    another workload or of an earlier version of the kernel source."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "k_gemm_mxf8_m1024_traffic.json")
    try:
        rec = json.load(open(path))["k_gemm_mxf8"]
        h = hashlib.sha256()
        for f in rec["source_files"]:
            h.update(open(os.path.join(ROOT, f), "rb").read())
    except (OSError, KeyError, ValueError):
        return None
    if h.hexdigest() != rec["source_sha256"] or workload != "m1024":
        return None
    return rec["dram_bytes_per_step"]


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
        self.marks = []

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

    def mark(self):
        self.marks.append(time.time())

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

    # ---- inputs, resident in HBM; R rotating sets so that the working set of
    # consecutive steps exceeds L2 (no flush needed between steps)
    x_h, w_h = wl.norm(seed=rank)
    a_h = {k: wl.gemm(k, seed=rank)[0] for k in ks}
    wt_h = {k: wl.gemm(k, seed=rank)[1] for k in ks}
    w_dev = w_h.to(dev)
    wq = {}
    for k in ks:
        wd = wt_h[k].to(dev)
        wq[k] = mx.quant(wd)
        del wd
    set_bytes = 2 * M * H + M * H + mx.mx_scale_bytes(M, H)
    for k in ks:
        set_bytes += 3 * M * k + mx.mx_scale_bytes(M, k) + 2 * M * N_OUT
    weight_bytes = sum(N_OUT * k + mx.mx_scale_bytes(N_OUT, k) for k in ks)
    R = max(2, math.ceil(2.2 * L2_BYTES / max(1, set_bytes + weight_bytes)))
    R = min(R, 16)
    sets = []
    for r in range(R):
        s = {"x": x_h.to(dev), "q": torch.empty((M, H), dtype=torch.uint8, device=dev),
             "s": torch.empty(mx.mx_scale_bytes(M, H), dtype=torch.uint8, device=dev)}
        for k in ks:
            s[f"a{k}"] = a_h[k].to(dev)
            s[f"aq{k}"] = torch.empty((M, k), dtype=torch.uint8, device=dev)
            s[f"as{k}"] = torch.empty(mx.mx_scale_bytes(M, k), dtype=torch.uint8, device=dev)
            s[f"c{k}"] = torch.empty((M, N_OUT), dtype=torch.bfloat16, device=dev)
        sets.append(s)
    # weights rotate too (each decoder layer has its own)
    wsets = [wq] + [{k: (wq[k][0].clone(), wq[k][1].clone()) for k in ks} for _ in range(R - 1)]
    torch.cuda.synchronize()

    def step(i, ev=None):
        s = sets[i % R]
        wsx = wsets[i % R]
        j = 0

        def mark():
            nonlocal j
            if ev is not None:
                ev[j].record(stream)
            j += 1

        mark()
        mx.mx_rmsnorm_quant(s["x"], w_dev, EPS, s["q"], s["s"], M, H, sptr)
        mark()
        for k in ks:
            mx.mx_quant_weights(s[f"a{k}"], s[f"aq{k}"], s[f"as{k}"], M, k, sptr)
            mark()
            mx.mx_gemm(s[f"aq{k}"], s[f"as{k}"], wsx[k][0], wsx[k][1], s[f"c{k}"], M, N_OUT, k, sptr)
            mark()

    def one_kernel(i, idx):
        s = sets[i % R]
        wsx = wsets[i % R]
        if idx == 0:
            mx.mx_rmsnorm_quant(s["x"], w_dev, EPS, s["q"], s["s"], M, H, sptr)
            return
        k = ks[(idx - 1) // 2]
        if (idx - 1) % 2 == 0:
            mx.mx_quant_weights(s[f"a{k}"], s[f"aq{k}"], s[f"as{k}"], M, k, sptr)
        else:
            mx.mx_gemm(s[f"aq{k}"], s[f"as{k}"], wsx[k][0], wsx[k][1], s[f"c{k}"], M, N_OUT, k, sptr)

    n_marks = 2 + 2 * len(ks)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    stream.synchronize()
    assert mx.mx_device_fault() == 0

    # The K timed steps are captured once as a CUDA graph (the launches go
    # through the same C entry points; the graph removes the host's per-call
    # launch latency, as a serving engine's CUDA-graph mode does).  For the
    # per-kernel breakdown each kernel of the step also gets a graph of its K
    # launches over the same rotating buffers, timed the same way.
    g_main = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_main, stream=stream):
        for i in range(args.steps):
            step(i)
    order = ["norm_quant"]
    for k in ks:
        order += [f"quant_a{k}", f"gemm_k{k}"]
    g_kern = []
    for idx in range(len(order)):
        gk = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gk, stream=stream):
            for i in range(args.steps):
                one_kernel(i, idx)
        g_kern.append(gk)
    torch.cuda.synchronize()

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    # soak ~1.5 s so the clocks under load are sampled and settled
    t_soak = time.time()
    with torch.cuda.stream(stream):
        while time.time() - t_soak < 1.5:
            for _ in range(5):
                g_main.replay()
            stream.synchronize()

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        g_main.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_wall1 = time.time()
    total_ms = e0.elapsed_time(e1)

    # per-kernel durations: each kernel's graph of K launches, replayed once
    per_kernel = {}
    with torch.cuda.stream(stream):
        for idx, name in enumerate(order):
            b0 = torch.cuda.Event(enable_timing=True)
            b1 = torch.cuda.Event(enable_timing=True)
            b0.record(stream)
            g_kern[idx].replay()
            b1.record(stream)
            stream.synchronize()
            per_kernel[name] = b0.elapsed_time(b1)
    breakdown_ms = sum(per_kernel.values())
    torch.cuda.synchronize()
    sampler.stop()
    assert mx.mx_device_fault() == 0
    ms_per_step = total_ms / args.steps

    flops_step = sum(gemm_flops(M, N_OUT, k) for k in ks)
    gemm_ms = sum(per_kernel[f"gemm_k{k}"] for k in ks)

    # ---- end to end through the C ABI with host buffers
    e2e = run_e2e(args, mx, torch, dev, stream, wl, x_h, w_dev, a_h, wq, ks)

    # ---- aggregate over ranks: max time, sum of work
    ms_max, value = aggregate_over_ranks(ms_per_step, flops_step / 1e12, world, dev)

    peaks = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_PER_BF16
    gemm_tflops = flops_step * args.steps / (gemm_ms * 1e-3) / 1e12
    nq_ms = per_kernel["norm_quant"] / args.steps
    nq_gbs = norm_quant_bytes(M) / (nq_ms * 1e-3) / 1e9
    kern = {}
    denom = breakdown_ms
    for name in order:
        ms = per_kernel[name] / args.steps
        if name == "norm_quant":
            b = norm_quant_bytes(M)
            kern[name] = {"us": ms * 1e3, "GB/s": b / (ms * 1e-3) / 1e9, "frac_hbm": b / (ms * 1e-3) / 1e9 /
                          peaks["hbm_gbs"], "share": per_kernel[name] / denom}
        elif name.startswith("quant_a"):
            k = int(name[7:])
            b = quant_bytes(M, k)
            kern[name] = {"us": ms * 1e3, "GB/s": b / (ms * 1e-3) / 1e9, "frac_hbm": b / (ms * 1e-3) / 1e9 /
                          peaks["hbm_gbs"], "share": per_kernel[name] / denom}
        else:
            k = int(name[6:])
            f = gemm_flops(M, N_OUT, k)
            kern[name] = {"us": ms * 1e3, "TFLOP/s": f / (ms * 1e-3) / 1e12,
                          "frac_fp8": f / (ms * 1e-3) / 1e12 / fp8_peak, "share": per_kernel[name] / denom}
    plan = {k: mx.mx_gemm_plan(M, N_OUT, k) for k in ks}

    clocks = sampler.summary(t_soak, t_wall1)
    out = {
        "metric": "MXFP8 GEMM TFLOP/s (% FP8 peak) & norm-quant GB/s, M=128-32768, N=6144",
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
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights, U(-0.1,0.1) norm gain)",
        "config": {"workload": wl.name, "M": M, "N": N_OUT, "K": list(ks), "norm_quant": f"{M}x{H}",
                   "step": "norm-quant(x) + per K: quant(A) + gemm(A, W_pre-quantised)",
                   "l2": f"{R} rotating input+weight sets, {(set_bytes + weight_bytes) * R / 2**20:.0f} MiB "
                         f"total > L2 (no flush)",
                   "parallelism": f"weak, {world} independent rank(s)", "gemm_plan": plan},
        "gemm_tflops": gemm_tflops,
        "norm_quant_gbs": nq_gbs,
        "kernels": kern,
        "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": gemm_tflops / fp8_peak, "traffic": gemm_traffic_per_step(args.workload),
                     "kernel": "k_gemm_mxf8 (both launches of the step)",
                     "peak_source": f"{peaks['source']} bf16 {peaks['bf16_tflops']} TFLOP/s x {FP8_PER_BF16} "
                                    "(nominal dense FP8/BF16 ratio)"},
        "norm_quant_roofline": {"bound": "hbm", "achieved": nq_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": nq_gbs / peaks["hbm_gbs"], "peak_source": peaks["source"]},
        "e2e": e2e,
        "gpu_launches": len(order) * args.steps,
        "timing": {"timed_region": "one CUDA-graph replay of the K steps (CUDA events on the launch stream)",
                   "per_kernel": "one CUDA graph of the kernel's K launches per kernel (same rotating buffers), "
                                 "CUDA events on the launch stream; shares are of the sum of these"},
        "clocks": clocks,
        "wall_s_timed": t_wall1 - t_wall0,
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        out["cpu_baseline"] = cpu_baseline(wl, ks, budget_s=args.cpu_seconds)
    return out


def run_e2e(args, mx, torch, dev, stream, wl, x_h, w_dev, a_h, wq, ks):
    """Same metric end to end: every step copies its inputs from pinned host
    memory to the device, runs the step through the C ABI and copies all of
    its outputs (codes, scales, C) back to pinned host memory.  Steps are
    pipelined as a serving loop runs them: copy-in, compute and copy-out on
    three streams with double-buffered device and host buffers, so step i's
    compute overlaps step i+1's copy-in and step i-1's copy-out.  The timed
    region runs from before the first copy-in to after the last copy-out."""
    M = wl.m
    x_pin = x_h.pin_memory()
    a_pin = {k: a_h[k].pin_memory() for k in ks}

    def buffers():
        b = {"x": torch.empty_like(x_pin, device=dev),
             "q": torch.empty((M, H), dtype=torch.uint8, device=dev),
             "s": torch.empty(mx.mx_scale_bytes(M, H), dtype=torch.uint8, device=dev)}
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
        mx.mx_rmsnorm_quant(b["x"], w_dev, EPS, b["q"], b["s"], M, H, sp)
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
    e1.record(s_out)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    flops = sum(gemm_flops(M, N_OUT, k) for k in ks)
    return {"value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipeline": "copy-in, compute and copy-out streams, double-buffered device and pinned host buffers"}


# ------------------------------------------------------------------ CPU oracle arm

def _oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count() or 1


def _oracle_prepare(wl, ks, rows):
    """Untimed: seeded inputs as the oracle takes them, weights quantised by the oracle."""
    import numpy as np
    import torch

    import oracle as O

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    x, w = wl.norm(seed=0)
    ops = []
    for k in ks:
        a, wt = wl.gemm(k, seed=0)
        bq, bs = O.quant(bits(wt))
        ops.append((k, bits(a[:rows]), bq, bs))
    return {"x": bits(x[:rows]), "w": bits(w), "ops": ops, "rows": rows}


def _oracle_step(prep):
    """One bounded sample of a step, run by the oracle as it stands: norm-quant
    of `rows` rows of x, quantisation of `rows` rows of each A, and their GEMM
    rows against the full 6144-row weight.  Returns the GEMM flops done."""
    import oracle as O
    O.rmsnorm_quant(prep["x"], prep["w"], EPS)
    flops = 0.0
    for k, ab, bq, bs in prep["ops"]:
        aq, as_ = O.quant(ab)
        O.gemm_ref(aq, as_, bq, bs)
        flops += gemm_flops(prep["rows"], N_OUT, k)
    return flops


def _sample_text(wl, ks, rows, n, dt):
    return (f"{n} x ({rows} rows of norm-quant {wl.m}x{H}; {rows} rows of quant + GEMM vs the full "
            f"6144-row weight for K={list(ks)}), {dt:.1f} s")


def cpu_baseline(wl, ks, budget_s=15.0, rows=16):
    """The oracle timed on a bounded row sample of the step, repeated for about
    budget_s seconds; reported as TFLOP/s of GEMM work."""
    prep = _oracle_prepare(wl, ks, rows)
    flops = 0.0
    n = 0
    t0 = time.time()
    while True:
        flops += _oracle_step(prep)
        n += 1
        if time.time() - t0 >= budget_s:
            break
    dt = time.time() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": _oracle_threads(), "kind": "oracle",
            "sample": _sample_text(wl, ks, rows, n, dt)}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, each step one bounded sample of the workload."""
    from mxfp8_norm_quant_gb300 import workloads as W
    wl = W.get_workload(args.workload)
    ks = wl.ks
    rows = 16
    prep = _oracle_prepare(wl, ks, rows)
    for _ in range(args.warmup):
        _oracle_step(prep)
    t0 = time.time()
    flops = 0.0
    for _ in range(args.steps):
        flops += _oracle_step(prep)
    dt = time.time() - t0
    value = flops / dt / 1e12
    return {
        "impl": "reference",
        "metric": "MXFP8 GEMM TFLOP/s (% FP8 peak) & norm-quant GB/s, M=128-32768, N=6144",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 GEMM of decoded MXFP8, f32 norm", "data": "synthetic",
        "config": {"workload": wl.name, "M": wl.m, "N": N_OUT, "K": list(ks), "norm_quant": f"{wl.m}x{H}",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": _oracle_threads(), "kind": "oracle",
                         "sample": _sample_text(wl, ks, rows, args.steps, dt)},
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
    ap.add_argument("--workload", default="m1024")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
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
