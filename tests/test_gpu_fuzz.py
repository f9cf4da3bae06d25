"""Seeded random shapes through every row kernel's dispatcher: the fused norm
in its three output forms and the plain quantiser, bit-exact against the
oracle.  Widths are multiples of 32 up to 16384 (multiples of 64 go to the
lane-block kernels, odd multiples of 32 to the chunked kernels), row counts
from 1 to a few thousand, and the inputs mix magnitudes, zero blocks and
outlier channels.

The seeds and the number of shapes can be raised for a longer campaign:
MX_FUZZ_SEED / MX_FUZZ_N (norm and quantiser shapes, default 2024 / 24) and
MX_FUZZ_GEMM_SEED / MX_FUZZ_GEMM_N (default 77 / 20)."""

import os

import numpy as np
import pytest
import torch

import mxfp8_norm_quant_gb300 as mx
import oracle as O
from mxfp8_norm_quant_gb300 import workloads as W
from mxtest import bf16_bits, np_u8

pytestmark = pytest.mark.gpu


def _shapes(seed, n):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        # half the widths near the models' width (4097..6144, % 64 == 0)
        if rng.random() < 0.5:
            h = int(rng.integers(65, 97)) * 64
        else:
            h = int(rng.integers(1, 513)) * 32
        m = int(rng.choice([1, 2, 3, 127, 129, 255, 300, 777, 1100, 2500, 3333]))
        out.append((m, h))
    return out


SHAPES = _shapes(int(os.environ.get("MX_FUZZ_SEED", "2024")), int(os.environ.get("MX_FUZZ_N", "24")))


def _inputs(m, h, seed):
    rng = np.random.default_rng(seed)
    x, w = W.norm_inputs(m, h, seed=seed, outlier_frac=0.01 if rng.random() < 0.5 else 0.0,
                         zero_block_frac=1 / 64 if rng.random() < 0.5 else 0.0)
    scale = float(np.exp2(rng.integers(-20, 21)))
    return (x.float() * scale).to(torch.bfloat16), w


@pytest.mark.parametrize("M,H", SHAPES, ids=[f"{m}x{h}" for m, h in SHAPES])
def test_fuzz_norm_forms(cuda_dev, M, H):
    x, w = _inputs(M, H, M * 131 + H)
    xb, wb = bf16_bits(x), bf16_bits(w)
    y = O.gemma_rmsnorm_f32(xb, wb, 1e-6)
    rq, rs_logical = O.mx_quantize_logical(y)
    xd, wd = x.to(cuda_dev), w.to(cuda_dev)
    q = torch.full((M, H), 0xA5, dtype=torch.uint8, device=cuda_dev)
    s = torch.full((mx.mx_scale_bytes(M, H),), 0xA5, dtype=torch.uint8, device=cuda_dev)
    mx.mx_rmsnorm_quant(xd, wd, 1e-6, q, s, M, H)
    qr = torch.full((M, H), 0xA5, dtype=torch.uint8, device=cuda_dev)
    sr = torch.full((M * (H // 32),), 0xA5, dtype=torch.uint8, device=cuda_dev)
    mx.mx_rmsnorm_quant_ex(xd, wd, 1e-6, qr, sr, M, H, mx.MX_SCALES_ROW_MAJOR)
    yd = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device=cuda_dev)
    mx.mx_rmsnorm_bf16(xd, wd, 1e-6, yd, M, H)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    assert np.array_equal(np_u8(q), rq)
    assert np.array_equal(np_u8(s), O.swizzle_scales(rs_logical))
    assert np.array_equal(np_u8(qr), rq)
    assert np.array_equal(np_u8(sr).reshape(M, -1), rs_logical)
    assert np.array_equal(bf16_bits(yd), O.f32_to_bf16_bits(y))


@pytest.mark.parametrize("M,H", SHAPES, ids=[f"{m}x{h}" for m, h in SHAPES])
def test_fuzz_quant(cuda_dev, M, H):
    x, _ = _inputs(M, H, M * 7 + H * 3)
    rq, rs = O.quant(bf16_bits(x))
    q = torch.full((M, H), 0xA5, dtype=torch.uint8, device=cuda_dev)
    s = torch.full((mx.mx_scale_bytes(M, H),), 0xA5, dtype=torch.uint8, device=cuda_dev)
    mx.mx_quant_weights(x.to(cuda_dev), q, s, M, H)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    assert np.array_equal(np_u8(q), rq)
    assert np.array_equal(np_u8(s), rs)


def _gemm_shapes(seed, n):
    rng = np.random.default_rng(seed)
    tiles = [(0, 0), (128, 64), (128, 128), (128, 192), (256, 128), (256, 192), (256, 256)]
    out = []
    for _ in range(n):
        m = int(rng.integers(1, 700))
        nn = int(rng.integers(1, 200)) * 32           # N % 32 == 0, so the MXFP8 output form applies too
        k = int(rng.integers(1, 80)) * 32             # K tails that are not a multiple of 128
        out.append((m, nn, k, tiles[int(rng.integers(0, len(tiles)))]))
    return out


GEMM_SHAPES = _gemm_shapes(int(os.environ.get("MX_FUZZ_GEMM_SEED", "77")), int(os.environ.get("MX_FUZZ_GEMM_N", "20")))


@pytest.mark.parametrize("M,N,K,tile", GEMM_SHAPES, ids=[f"{m}x{n}x{k}-{t[0]}x{t[1]}" for m, n, k, t in GEMM_SHAPES])
def test_fuzz_gemm(cuda_dev, M, N, K, tile):
    # random shapes: ragged M and N tiles and K tails, every tile; the bf16
    # output against the float64 oracle within the GEMM tolerance, and the
    # MXFP8 output equal to the quantiser applied to that bf16 output
    from mxtest import gemm_close
    a, wt = W.gemm_operands(M, K, seed=M + 3 * N + 7 * K, n=N)
    aq, as_ = O.quant(bf16_bits(a))
    bq, bs_ = O.quant(bf16_bits(wt))
    d = [torch.from_numpy(np.ascontiguousarray(t)).to(cuda_dev) for t in (aq, as_, bq, bs_)]
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=cuda_dev)
    mx.mx_gemm_ex(*d, out, M, N, K, *tile)
    q = torch.full((M, N), 0xA5, dtype=torch.uint8, device=cuda_dev)
    s = torch.full((mx.mx_scale_bytes(M, N),), 0xA5, dtype=torch.uint8, device=cuda_dev)
    mx.mx_gemm_quant(*d, q, s, M, N, K, *tile)
    cq, cs = mx.quant(out)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    ok, worst = gemm_close(out, O.gemm_ref(aq, as_, bq, bs_))
    assert ok, f"worst err/tol = {worst:.3f}"
    if tile != (0, 0):
        # the same tile's accumulators: the fused epilogue equals the plain quantiser
        assert torch.equal(q, cq) and torch.equal(s, cs)
