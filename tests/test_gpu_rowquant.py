"""GPU parity of mx_rmsnorm_quant and mx_quant_weights against the oracle:
E4M3 codes and the whole F8_128x4 scale buffer (padding included) must match
bit for bit."""

import numpy as np
import pytest
import torch

import mxfp8_norm_quant_gb300 as mx
import oracle as O
from mxfp8_norm_quant_gb300 import workloads as W
from mxtest import bf16_bits, np_u8

pytestmark = pytest.mark.gpu


def _run_norm(x, w, eps, dev):
    M, H = x.shape
    xd, wd = x.to(dev), w.to(dev)
    q = torch.full((M, H), 0xA5, dtype=torch.uint8, device=dev)        # poison: every byte must be written
    s = torch.full((mx.mx_scale_bytes(M, H),), 0xA5, dtype=torch.uint8, device=dev)
    mx.mx_rmsnorm_quant(xd, wd, eps, q, s, M, H)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    return np_u8(q), np_u8(s)


def _run_quant(x, dev):
    R, C = x.shape
    q = torch.full((R, C), 0xA5, dtype=torch.uint8, device=dev)
    s = torch.full((mx.mx_scale_bytes(R, C),), 0xA5, dtype=torch.uint8, device=dev)
    mx.mx_quant_weights(x.to(dev), q, s, R, C)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    return np_u8(q), np_u8(s)


def _assert_same(got_q, got_s, ref_q, ref_s):
    bad = np.argwhere(got_q != ref_q)
    assert bad.size == 0, f"{len(bad)} code mismatches, first at {bad[:5].tolist()}"
    bad_s = np.flatnonzero(got_s != ref_s)
    assert bad_s.size == 0, f"{bad_s.size} scale-byte mismatches, first offsets {bad_s[:8].tolist()}"


SMALL = [(1, 32), (3, 96), (127, 256), (128, 384), (130, 2048), (300, 6144), (64, 6176), (129, 6144),
         (2, 8192), (33, 9984), (5, 16384), (257, 160)]


@pytest.mark.parametrize("M,H", SMALL)
def test_norm_quant_small(cuda_dev, M, H):
    x, w = W.norm_inputs(M, H, seed=M * 7 + H)
    rq, rs = O.rmsnorm_quant(bf16_bits(x), bf16_bits(w), 1e-6)
    _assert_same(*_run_norm(x, w, 1e-6, cuda_dev), rq, rs)


# Row counts at H = 6144 on either side of each kernel choice of the
# dispatcher on a 152-SM GPU: 6 warps per row (<= 256 rows), 3 warps per row
# (<= 760), the prefetching kernel (>= 761; the row-major form keeps 6 warps
# per row below 896), and its reduce-scatter sum of squares (1217-9728 rows).
# Every variant must give the same bytes.
DISPATCH_ROWS = [256, 257, 760, 761, 895, 896, 1216, 1217, 9728, 9729]


@pytest.mark.parametrize("M", DISPATCH_ROWS)
def test_norm_quant_dispatch_boundaries(cuda_dev, M):
    H = 6144
    x, w = W.norm_inputs(M, H, seed=M + 11)
    rq, rs = O.rmsnorm_quant(bf16_bits(x), bf16_bits(w), 1e-6)
    _assert_same(*_run_norm(x, w, 1e-6, cuda_dev), rq, rs)


@pytest.mark.parametrize("M,H", SMALL)
def test_quant_small(cuda_dev, M, H):
    x = W.normal_bf16((M, H), 1.0, seed=M + H, tag="A")
    rq, rs = O.quant(bf16_bits(x))
    _assert_same(*_run_quant(x, cuda_dev), rq, rs)


def test_norm_quant_degenerate_rows(cuda_dev):
    # all-zero rows (r = 1/sqrt(eps)), constant rows, huge and tiny magnitudes,
    # subnormal bf16 inputs, zero blocks, gain w = -1 (y = 0) and w large
    M, H = 256, 6144
    x, w = W.norm_inputs(M, H, seed=3)
    x = x.float()
    x[0] = 0.0
    x[1] = 1.0
    x[2] *= 1e30
    x[3] *= 1e-30
    x[4] = 2.0 ** -133
    x[5, :32] = 0.0
    x[6, ::2] = -0.0
    x[7, 100] = 3e38
    x = x.to(torch.bfloat16)
    w = w.float()
    w[:64] = -1.0
    w[64:96] = 7.5
    w = w.to(torch.bfloat16)
    for eps in (1e-6, 0.0, 1.0):
        if eps == 0.0:
            # rows whose squares all underflow give r = 1/0 and y = NaN: outside
            # the domain, so with eps = 0 they are replaced by ones
            xx = x.clone()
            xx[0] = 1.0
            xx[3] = 1.0
            xx[4] = 1.0
        else:
            xx = x
        rq, rs = O.rmsnorm_quant(bf16_bits(xx), bf16_bits(w), eps)
        _assert_same(*_run_norm(xx, w, eps, cuda_dev), rq, rs)


def test_quant_every_bf16_pattern(cuda_dev):
    # every finite bf16 bit pattern, in blocks that mix magnitudes
    bits = np.arange(1 << 16, dtype=np.uint32)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    vals = bits[finite].astype(np.uint16)
    rng = np.random.default_rng(0)
    vals = rng.permutation(vals)
    n = (vals.size // 256) * 256
    x = torch.from_numpy(vals[:n].view(np.int16).copy()).view(torch.bfloat16).reshape(-1, 256)
    rq, rs = O.quant(bf16_bits(x))
    _assert_same(*_run_quant(x, cuda_dev), rq, rs)
    # the same patterns sorted, so that whole blocks share one binade
    xs = torch.from_numpy(np.sort(vals[:n]).view(np.int16).copy()).view(torch.bfloat16).reshape(-1, 256)
    rq, rs = O.quant(bf16_bits(xs))
    _assert_same(*_run_quant(xs, cuda_dev), rq, rs)


def test_zero_rows_is_noop(cuda_dev):
    q = torch.full((4,), 7, dtype=torch.uint8, device=cuda_dev)
    mx.mx_rmsnorm_quant(q, q, 1e-6, q, q, 0, 64)
    mx.mx_quant_weights(q, q, q, 0, 64)
    torch.cuda.synchronize()
    assert torch.all(q == 7)


@pytest.mark.parametrize("name", ["m128", "m1024", "m4096_rowscale"])
def test_norm_quant_workloads_full(cuda_dev, name):
    wl = W.WORKLOADS[name]
    x, w = wl.norm()
    rq, rs = O.rmsnorm_quant(bf16_bits(x), bf16_bits(w), wl.eps)
    _assert_same(*_run_norm(x, w, wl.eps, cuda_dev), rq, rs)


def test_norm_quant_stress_full_size(cuda_dev):
    # 32768 x 6144 residual with outlier channels and zero blocks, in the
    # launch configuration the bench times: every row's codes and the whole
    # F8_128x4 scale buffer (padding included) against the oracle, which runs
    # over row chunks of 4096 (a multiple of 128, so each chunk's swizzled
    # scales are one contiguous span of the full buffer)
    wl = W.WORKLOADS["m32768_stress"]
    x, w = wl.norm()
    M, H = x.shape
    gq, gs = _run_norm(x, w, wl.eps, cuda_dev)
    xb, wb = bf16_bits(x), bf16_bits(w)
    span = O.scale_bytes(4096, H)
    for r in range(0, M, 4096):
        rq, rs = O.rmsnorm_quant(xb[r:r + 4096], wb, wl.eps)
        _assert_same(gq[r:r + 4096], gs[r // 4096 * span:(r // 4096 + 1) * span], rq, rs)
    assert gs.size == (M // 4096) * span
    # row 0 is all zero: scale bytes 0 and codes 0
    c = H // 32
    assert np.all(gq[0] == 0) and np.all(O.unswizzle_scales(gs, 1, c) == 0)
    # the stressors really exercised saturation (codes 0x7E / 0xFE) and zero blocks
    assert np.any((gq & 0x7F) == 0x7E)


@pytest.mark.parametrize("k", [W.K_OPROJ, W.K_DOWN])
def test_quant_weights_full(cuda_dev, k):
    wl = W.WORKLOADS["m4096_rowscale"]
    a, wt = wl.gemm(k)
    for t in (a, wt):
        rq, rs = O.quant(bf16_bits(t))
        _assert_same(*_run_quant(t, cuda_dev), rq, rs)
