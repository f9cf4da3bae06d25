"""Concurrency and graph capture through the C ABI.

* Several host threads, each with its own CUDA stream, call the library at
  once (the header promises thread safety: per-device set-up runs once, the
  shared-memory attribute table is locked, the cluster-occupancy cache is
  atomic).  Every thread's results must equal the single-threaded ones.
* A whole step (norm-quant, operand quantisation, GEMM, MXFP8-output GEMM)
  captured in a CUDA graph and replayed must give the bytes the eager calls
  give (the tensor maps are encoded at capture time from the buffers the
  graph will use).
* The norm's output fed straight into a GEMM, and overwritten by the next
  norm, back to back on one stream: the dependent-launch waits must order
  each read before the next write."""

import threading

import numpy as np
import pytest
import torch

import mxfp8_norm_quant_gb300 as mx
import oracle as O
from mxfp8_norm_quant_gb300 import workloads as W
from mxtest import bf16_bits, gemm_close, np_u8

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


def test_norm_codes_feed_the_gemm_back_to_back(cuda_dev):
    # the norm's MXFP8 output is the A operand of a GEMM (K = H), and the next
    # norm overwrites the same q / s while that GEMM may still be reading them:
    # launched back to back on one stream with no host synchronisation, each
    # kernel's dependent-launch wait must order the read before the overwrite
    M, H, N = 640, 6144, 1536
    st = torch.cuda.Stream(cuda_dev)
    _, wt = W.gemm_operands(16, H, seed=3, n=N)
    bq, bs_ = mx.quant(wt.to(cuda_dev))
    q = torch.empty((M, H), dtype=torch.uint8, device=cuda_dev)
    s = torch.empty(mx.mx_scale_bytes(M, H), dtype=torch.uint8, device=cuda_dev)
    xs, ws, cs = [], [], []
    for i in range(4):
        x, w = W.norm_inputs(M, H, seed=40 + i, outlier_frac=0.01)
        xs.append(x)
        ws.append(w)
    xd = [x.to(cuda_dev) for x in xs]
    wd = [w.to(cuda_dev) for w in ws]
    torch.cuda.synchronize()
    sp = st.cuda_stream
    for i in range(4):
        c = torch.empty((M, N), dtype=torch.bfloat16, device=cuda_dev)
        mx.mx_rmsnorm_quant(xd[i], wd[i], 1e-6, q, s, M, H, sp)
        mx.mx_gemm(q, s, bq, bs_, c, M, N, H, sp)
        cs.append(c)
    st.synchronize()
    assert mx.mx_device_fault() == 0
    rows = np.arange(0, M, 5)
    for i in range(4):
        rq, rs = O.rmsnorm_quant(bf16_bits(xs[i]), bf16_bits(ws[i]), 1e-6)
        a_rows = O.swizzle_scales(O.unswizzle_scales(rs, M, H // 32)[rows])
        ref = O.gemm_ref(rq[rows], a_rows, np_u8(bq), np_u8(bs_))
        ok, worst = gemm_close(cs[i][torch.from_numpy(rows).to(cuda_dev)], ref)
        assert ok, f"launch {i}: worst err/tol = {worst:.3f}"
