"""Seeded random shapes through every row kernel's dispatcher: the fused norm
in its three output forms and the plain quantiser, bit-exact against the
oracle.  Widths are multiples of 32 up to 16384 (both the lane-block kernels'
range and the chunked kernels'), row counts from 1 to a few thousand, and the
inputs mix magnitudes, zero blocks and outlier channels."""

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
        # half the widths in the lane-block kernels' range (4097..6144, % 64 == 0)
        if rng.random() < 0.5:
            h = int(rng.integers(65, 97)) * 64
        else:
            h = int(rng.integers(1, 513)) * 32
        m = int(rng.choice([1, 2, 3, 127, 129, 255, 300, 777, 1100, 2500, 3333]))
        out.append((m, h))
    return out


SHAPES = _shapes(2024, 24)


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
