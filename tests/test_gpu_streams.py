"""Concurrency and graph capture through the C ABI.

* Several host threads, each with its own CUDA stream, call the library at
  once (the header promises thread safety: per-device set-up runs once, the
  shared-memory attribute table is locked, the cluster-occupancy cache is
  atomic).  Every thread's results must equal the single-threaded ones.
* A whole step (norm-quant, operand quantisation, GEMM, MXFP8-output GEMM)
  captured in a CUDA graph and replayed must give the bytes the eager calls
  give (the tensor maps are encoded at capture time from the buffers the
  graph will use)."""

import threading

import pytest
import torch

import mxfp8_norm_quant_gb300 as mx
from mxfp8_norm_quant_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _step(x, w, a, wq, M, H, K, stream):
    """One pass of the path on `stream`; returns its outputs (allocated here)."""
    dev = x.device
    sp = stream.cuda_stream
    q = torch.empty((M, H), dtype=torch.uint8, device=dev)
    s = torch.empty(mx.mx_scale_bytes(M, H), dtype=torch.uint8, device=dev)
    aq = torch.empty((M, K), dtype=torch.uint8, device=dev)
    as_ = torch.empty(mx.mx_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    c = torch.empty((M, 6144), dtype=torch.bfloat16, device=dev)
    cq = torch.empty((M, 6144), dtype=torch.uint8, device=dev)
    cs = torch.empty(mx.mx_scale_bytes(M, 6144), dtype=torch.uint8, device=dev)
    mx.mx_rmsnorm_quant(x, w, 1e-6, q, s, M, H, sp)
    mx.mx_quant_weights(a, aq, as_, M, K, sp)
    mx.mx_gemm(aq, as_, wq[0], wq[1], c, M, 6144, K, sp)
    mx.mx_gemm_quant(aq, as_, wq[0], wq[1], cq, cs, M, 6144, K, 0, 0, sp)
    return q, s, aq, as_, c, cq, cs


def _inputs(dev, M, K, seed):
    x, w = W.norm_inputs(M, 6144, seed=seed)
    a, wt = W.gemm_operands(M, K, seed=seed)
    wq = mx.quant(wt.to(dev))
    torch.cuda.synchronize()
    return x.to(dev), w.to(dev), a.to(dev), wq


@pytest.mark.parametrize("M,K", [(768, 2048), (1500, 3072)])
def test_threads_and_streams(cuda_dev, M, K):
    ref_in = _inputs(cuda_dev, M, K, seed=5)
    s0 = torch.cuda.Stream(cuda_dev)
    ref = _step(*ref_in, M, 6144, K, s0)
    torch.cuda.synchronize()
    errors = []
    results = {}

    def worker(t):
        try:
            torch.cuda.set_device(cuda_dev)
            st = torch.cuda.Stream(cuda_dev)
            outs = []
            for _ in range(6):
                outs.append(_step(*ref_in, M, 6144, K, st))
            st.synchronize()
            results[t] = outs
        except Exception as e:  # surfaced in the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(120)
    torch.cuda.synchronize()
    assert not errors, errors
    assert mx.mx_device_fault() == 0
    for t in range(4):
        for outs in results[t]:
            for got, want in zip(outs, ref):
                assert torch.equal(got, want)


def test_graph_capture_replays_eager_bytes(cuda_dev):
    M, K = 1024, 3072
    x, w, a, wq = _inputs(cuda_dev, M, K, seed=9)
    st = torch.cuda.Stream(cuda_dev)
    eager = _step(x, w, a, wq, M, 6144, K, st)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        graphed = _step(x, w, a, wq, M, 6144, K, st)
    for _ in range(3):
        for t in graphed:
            t.zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            g.replay()
        st.synchronize()
        for got, want in zip(graphed, eager):
            assert torch.equal(got, want)
    assert mx.mx_device_fault() == 0
