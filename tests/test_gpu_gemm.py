"""GPU parity of mx_gemm against the oracle's float64 GEMM of the decoded
operands: exact special cases (which also pin the scale layout), random
operands within |gpu - ref| <= 1e-2 (|ref| + 1) for every tile width and
ragged shapes, and the full-size workloads on sampled rows."""

import numpy as np
import pytest
import torch

import mxfp8_norm_quant_gb300 as mx
import oracle as O
from mxfp8_norm_quant_gb300 import workloads as W
from mxtest import bf16_bits, gemm_close, np_u8, to_dev

pytestmark = pytest.mark.gpu

TILES = [(128, 64), (128, 128), (128, 192), (256, 128), (256, 192), (256, 256)]


def _tid(t):
    return "auto" if t == (0, 0) else f"{t[0]}x{t[1]}"


def _gemm(aq, as_, bq, bs, M, N, K, dev, tile=(0, 0)):
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    mx.mx_gemm_ex(to_dev(aq, dev), to_dev(as_, dev), to_dev(bq, dev), to_dev(bs, dev), out, M, N, K, *tile)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    return out


def _random_codes(rng, shape):
    q = rng.integers(0, 256, size=shape, dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x38                    # no NaN codes
    return q


@pytest.mark.parametrize("tile", TILES, ids=_tid)
def test_one_hot_b_selects_a_elements(cuda_dev, tile):
    # B row n = E4M3 1.0 at column k_n (scale byte 127): C[m, n] = dec(A)[m, k_n]
    # exactly (4 significant bits fit bf16).  A's scale bytes vary by row and
    # K-block, so a misplaced scale or row fails.
    rng = np.random.default_rng(tile[0] + tile[1])
    M, N, K = 384, 448, 512
    aq = _random_codes(rng, (M, K))
    asb = rng.integers(110, 145, size=(M, K // 32), dtype=np.uint8)
    kn = rng.integers(0, K, size=N)
    bq = np.zeros((N, K), dtype=np.uint8)
    bq[np.arange(N), kn] = 0x38
    bsb = np.full((N, K // 32), 127, dtype=np.uint8)
    ref = O.gemm_ref(aq, O.swizzle_scales(asb), bq, O.swizzle_scales(bsb))
    got = _gemm(aq, O.swizzle_scales(asb), bq, O.swizzle_scales(bsb), M, N, K, cuda_dev, tile)
    expect = torch.from_numpy(ref).float().to(torch.bfloat16)
    assert torch.equal(got.cpu(), expect)


@pytest.mark.parametrize("tile", TILES, ids=_tid)
def test_small_integers_exact(cuda_dev, tile):
    # entries in {-1, 0, 1} x power-of-two scales that differ per row and
    # K-block of both operands: every partial sum is exact, so the bf16
    # output is the RNE rounding of the exact result, bit for bit.
    rng = np.random.default_rng(100 + tile[0] + tile[1])
    M, N, K = 384, 320, 640
    ai = rng.integers(-1, 2, size=(M, K))
    bi = rng.integers(-1, 2, size=(N, K))
    aq = O.e4m3_encode(ai.astype(np.float32))
    bq = O.e4m3_encode(bi.astype(np.float32))
    # scales x1/x2 on A and x0.5/x1 on B: |partial sums| <= 1280 at a granularity
    # of 0.5 (12 significant bits), exact even in a narrower accumulator
    asb = rng.integers(127, 129, size=(M, K // 32), dtype=np.uint8)
    bsb = rng.integers(126, 128, size=(N, K // 32), dtype=np.uint8)
    ref = O.gemm_ref(aq, O.swizzle_scales(asb), bq, O.swizzle_scales(bsb))
    got = _gemm(aq, O.swizzle_scales(asb), bq, O.swizzle_scales(bsb), M, N, K, cuda_dev, tile)
    expect = torch.from_numpy(ref).float().to(torch.bfloat16)
    assert torch.equal(got.cpu(), expect)


SHAPES = [(128, 6144, 2048), (1, 96, 32), (300, 416, 288), (129, 256, 4096), (512, 1024, 3072), (77, 6144, 160),
          (1000, 2016, 1024), (300, 512, 16384),
          # N % 32 == 16: the last 32-column chunk of C is half in the output
          (200, 48, 256), (130, 6160, 1024), (64, 16, 64)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("tile", [(0, 0)] + TILES, ids=_tid)
def test_random_within_tolerance(cuda_dev, M, N, K, tile):
    a, wt = W.gemm_operands(M, K, seed=M + N + K, n=N)
    aq, as_ = O.quant(bf16_bits(a))
    bq, bs_ = O.quant(bf16_bits(wt))
    ref = O.gemm_ref(aq, as_, bq, bs_)
    got = _gemm(aq, as_, bq, bs_, M, N, K, cuda_dev, tile)
    ok, worst = gemm_close(got, ref)
    assert ok, f"worst err/tol = {worst:.3f}"


@pytest.mark.parametrize("tile", [(128, 192), (256, 192)], ids=_tid)
def test_output_16_byte_aligned_only(cuda_dev, tile):
    # an output base that is 16- but not 32-byte aligned takes the 16-byte store path
    M, N, K = 300, 448, 256
    a, wt = W.gemm_operands(M, K, seed=5, n=N)
    aq, as_ = O.quant(bf16_bits(a))
    bq, bs_ = O.quant(bf16_bits(wt))
    ref = O.gemm_ref(aq, as_, bq, bs_)
    big = torch.full((M * N + 16,), float("nan"), dtype=torch.bfloat16, device=cuda_dev)
    base = big.data_ptr()
    off = 8 if (base + 16) % 32 else 16            # elements: 16 bytes past a 32-byte boundary
    out = big[off:off + M * N].view(M, N)
    assert out.data_ptr() % 32 == 16
    mx.mx_gemm_ex(to_dev(aq, cuda_dev), to_dev(as_, cuda_dev), to_dev(bq, cuda_dev), to_dev(bs_, cuda_dev), out,
                  M, N, K, *tile)
    torch.cuda.synchronize()
    ok, worst = gemm_close(out, ref)
    assert ok, f"worst err/tol = {worst:.3f}"


def test_zero_m_is_noop(cuda_dev):
    out = torch.full((4,), 3.0, dtype=torch.bfloat16, device=cuda_dev)
    mx.mx_gemm(0, 0, 0, 0, out, 0, 6144, 2048)
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)


def _workload_check(wl, k, dev, n_rows=256, seed=0):
    """The full-size GEMM exactly as bench.py launches it (operands quantised by
    the GPU kernels, which are themselves checked bit-exact elsewhere), checked
    against the oracle on a row sample, or on every row when n_rows is None
    (the oracle then runs over row chunks of 4096)."""
    a, wt = wl.gemm(k, seed)
    M, N = a.shape[0], wt.shape[0]
    ad, wd = a.to(dev), wt.to(dev)
    aq, as_ = mx.quant(ad)
    bq, bs_ = mx.quant(wd)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    mx.mx_gemm(aq, as_, bq, bs_, out, M, N, k)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    # operands for the oracle: from the oracle's own quantiser
    bq_o, bs_o = O.quant(bf16_bits(wt))
    if n_rows is None or n_rows >= M:
        worst = 0.0
        ab = bf16_bits(a)
        for r in range(0, M, 4096):
            aq_o, as_o = O.quant(ab[r:r + 4096])
            ok, w_ = gemm_close(out[r:r + 4096], O.gemm_ref(aq_o, as_o, bq_o, bs_o))
            assert ok, f"{wl.name} K={k} rows {r}..: worst err/tol = {w_:.3f}"
            worst = max(worst, w_)
        return worst
    rng = np.random.default_rng(seed + M + k)
    rows = np.unique(np.concatenate([[0, M - 1], rng.choice(M, min(M, n_rows), replace=False)]))
    aq_o, as_o = O.quant(bf16_bits(a[torch.from_numpy(rows)]))
    ref = O.gemm_ref(aq_o, as_o, bq_o, bs_o)
    ok, worst = gemm_close(out[torch.from_numpy(rows).to(dev)], ref)
    assert ok, f"{wl.name} K={k}: worst err/tol = {worst:.3f}"
    return worst


@pytest.mark.parametrize("name,k", [("m128", 2048), ("m1024", 2048), ("m1024", 3072), ("m4096_rowscale", 2048),
                                    ("m4096_rowscale", 3072), ("m32768_stress", 3072)])
def test_workload_full_size_every_element(cuda_dev, name, k):
    _workload_check(W.WORKLOADS[name], k, cuda_dev, n_rows=None)


@pytest.mark.parametrize("m", W.M_SWEEP)
@pytest.mark.parametrize("k", [W.K_OPROJ, W.K_DOWN])
def test_m_sweep(cuda_dev, m, k):
    # every element up to M = 4096, a 1024-row sample beyond
    _workload_check(W.sweep_workload(m, k), k, cuda_dev, n_rows=None if m <= 4096 else 1024, seed=1)


def test_plan_is_consistent(cuda_dev):
    for m in W.M_SWEEP:
        p = mx.mx_gemm_plan(m, 6144, 2048)
        assert (p["tile_m"], p["tile_n"]) in TILES and p["stages"] >= 2 and p["grid"] >= 1
