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


# Row counts on either side of each kernel choice of the chunked kernels'
# dispatcher on a 152-SM GPU, at H = 6112 (a width the lane-block kernels do
# not take): 6 warps per row (<= 256 rows), 3 warps per row (<= 760), the
# prefetching kernel (>= 761; the row-major form keeps 6 warps per row below
# 896), and its reduce-scatter sum of squares (1217-9728 rows).  Every
# variant must give the same bytes.
DISPATCH_ROWS = [256, 257, 760, 761, 895, 896, 1216, 1217, 9728, 9729]


@pytest.mark.parametrize("M", DISPATCH_ROWS)
def test_norm_quant_dispatch_boundaries(cuda_dev, M):
    H = 6112
    x, w = W.norm_inputs(M, H, seed=M + 11)
    rq, rs = O.rmsnorm_quant(bf16_bits(x), bf16_bits(w), 1e-6)
    _assert_same(*_run_norm(x, w, 1e-6, cuda_dev), rq, rs)


def lane_block_boundaries(num_sms):
    """Row counts on both sides of each kernel choice of the lane-block
    dispatcher (rows of 4097..6144 elements, H % 64 == 0), for this GPU's SM
    count: <6,1,2> up to 1.7 rows per SM, <3,2,5> to 4.65, <3,2,8> to 8,
    <3,2,5> to 16, then <3,2,8> and from 64 rows per SM <3,2,6> (the BF16
    form: <6,1,4> from 40.4 rows per SM)."""
    s = num_sms
    rows = []
    for last in (17 * s // 10, 465 * s // 100, 8 * s, 16 * s, 64 * s - 1, (202 * s - 1) // 5):
        rows += [last, last + 1]
    return rows


@pytest.mark.parametrize("i", range(12))
def test_norm_quant_lane_block_boundaries(cuda_dev, i):
    M = lane_block_boundaries(torch.cuda.get_device_properties(cuda_dev).multi_processor_count)[i]
    H = 6144
    x, w = W.norm_inputs(M, H, seed=M + 13, outlier_frac=0.01, zero_block_frac=1 / 128)
    rq, rs = O.rmsnorm_quant(bf16_bits(x), bf16_bits(w), 1e-6)
    _assert_same(*_run_norm(x, w, 1e-6, cuda_dev), rq, rs)


# lane-block kernels at widths whose last 1024-element chunk is partial
# (4160: 64 elements, and with 6 warps per row a warp with no chunk at all;
# 5184; 6080) or whole (5120), with ragged 128-row blocks
LB_SHAPES = [(300, 4160), (1000, 4160), (4000, 4160), (77, 5120), (3000, 5184), (129, 6080), (2000, 6080)]


@pytest.mark.parametrize("M,H", LB_SHAPES)
def test_norm_quant_lane_block_widths(cuda_dev, M, H):
    x, w = W.norm_inputs(M, H, seed=M * 5 + H)
    rq, rs = O.rmsnorm_quant(bf16_bits(x), bf16_bits(w), 1e-6)
    _assert_same(*_run_norm(x, w, 1e-6, cuda_dev), rq, rs)


@pytest.mark.parametrize("M,H", SMALL)
def test_quant_small(cuda_dev, M, H):
    x = W.normal_bf16((M, H), 1.0, seed=M + H, tag="A")
    rq, rs = O.quant(bf16_bits(x))
    _assert_same(*_run_quant(x, cuda_dev), rq, rs)


@pytest.mark.parametrize("M,H", [(256, 6144), (2000, 6144), (256, 6112), (1000, 4160), (3000, 512), (300, 1024),
                                 (700, 2048), (200, 3072), (1500, 4096), (300, 8192), (100, 16384)])
def test_norm_quant_degenerate_rows(cuda_dev, M, H):
    # all-zero rows (r = 1/sqrt(eps)), constant rows, huge and tiny magnitudes,
    # subnormal bf16 inputs, zero blocks, gain w = -1 (y = 0) and w large;
    # through the lane-block kernels (H = 6144, 4160 and one configuration of
    # each other width class) and the chunked ones (H = 6112)
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


def test_quant_every_bf16_pattern_lane_block(cuda_dev):
    # every finite bf16 pattern again, tiled into 1536 rows of 1024 elements:
    # enough 1024-element tasks to take the lane-block quantiser
    bits = np.arange(1 << 16, dtype=np.uint32)
    vals = bits[((bits >> 7) & 0xFF) != 0xFF].astype(np.uint16)
    vals = np.random.default_rng(2).permutation(vals)
    tiled = np.resize(vals, 1536 * 1024).reshape(1536, 1024)
    x = torch.from_numpy(tiled.view(np.int16).copy()).view(torch.bfloat16)
    rq, rs = O.quant(bf16_bits(x))
    _assert_same(*_run_quant(x, cuda_dev), rq, rs)


@pytest.mark.parametrize("K", [2048, 3072, 6144, 1056])
@pytest.mark.parametrize("side", [0, 1])
def test_quant_dispatch_boundary(cuda_dev, K, side):
    # the row counts on both sides of the switch from the chunked quantiser to
    # the lane-block one (10 tasks of 1024 elements per SM), plus a width
    # whose last chunk holds one block
    s = torch.cuda.get_device_properties(cuda_dev).multi_processor_count
    per_row = -(-K // 1024)
    M = -(-10 * s // per_row) - 1 + side
    x = W.normal_bf16((M, K), 1.0, seed=M + K, tag="A")
    rq, rs = O.quant(bf16_bits(x))
    _assert_same(*_run_quant(x, cuda_dev), rq, rs)


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
