"""Soak: the whole path replayed for a while must keep giving the same bytes.

Every kernel here is deterministic (fixed summation orders, one tile shape per
call), so a step captured in a CUDA graph and replayed thousands of times
must reproduce its first replay's outputs exactly; a rare race (an mbarrier
phase confused after many wraps, a copy overwriting a stage still being read)
would show up as a changed byte or a set fault bit.  The run length is
MX_SOAK_S seconds (default 5)."""

import os
import time

import pytest
import torch

import mxfp8_norm_quant_gb300 as mx
from mxfp8_norm_quant_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K", [(1024, 3072), (4096, 2048)])
def test_replayed_step_keeps_its_bytes(cuda_dev, M, K):
    H, N = 6144, 6144
    x, w = W.norm_inputs(M, H, seed=M + K, outlier_frac=0.01, zero_block_frac=1 / 128)
    a, wt = W.gemm_operands(M, K, seed=M + K)
    xd, wd, ad = x.to(cuda_dev), w.to(cuda_dev), a.to(cuda_dev)
    bq, bs_ = mx.quant(wt.to(cuda_dev))
    q = torch.empty((M, H), dtype=torch.uint8, device=cuda_dev)
    s = torch.empty(mx.mx_scale_bytes(M, H), dtype=torch.uint8, device=cuda_dev)
    aq = torch.empty((M, K), dtype=torch.uint8, device=cuda_dev)
    as_ = torch.empty(mx.mx_scale_bytes(M, K), dtype=torch.uint8, device=cuda_dev)
    c = torch.empty((M, N), dtype=torch.bfloat16, device=cuda_dev)
    cq = torch.empty((M, N), dtype=torch.uint8, device=cuda_dev)
    cs = torch.empty(mx.mx_scale_bytes(M, N), dtype=torch.uint8, device=cuda_dev)
    st = torch.cuda.Stream(cuda_dev)
    sp = st.cuda_stream
    torch.cuda.synchronize()

    def step():
        mx.mx_rmsnorm_quant(xd, wd, 1e-6, q, s, M, H, sp)
        mx.mx_quant_weights(ad, aq, as_, M, K, sp)
        mx.mx_gemm(aq, as_, bq, bs_, c, M, N, K, sp)
        mx.mx_gemm_quant(aq, as_, bq, bs_, cq, cs, M, N, K, 0, 0, sp)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for _ in range(8):
            step()
    with torch.cuda.stream(st):
        g.replay()
    st.synchronize()
    assert mx.mx_device_fault() == 0
    first = [t.clone() for t in (q, s, aq, as_, c, cq, cs)]
    seconds = float(os.environ.get("MX_SOAK_S", "5"))
    t_end = time.time() + seconds
    replays = 0
    while time.time() < t_end:
        for t in (q, s, aq, as_, c, cq, cs):
            t.zero_()
        with torch.cuda.stream(st):
            for _ in range(50):
                g.replay()
        st.synchronize()
        replays += 50
        assert mx.mx_device_fault() == 0, f"fault after {replays} replays"
        for got, want in zip((q, s, aq, as_, c, cq, cs), first):
            assert torch.equal(got, want), f"bytes changed after {replays} replays"
    assert replays > 0
