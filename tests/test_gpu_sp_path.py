"""GPU parity of the sequence-parallel forms of the norm (vLLM PR #65496,
Details / Tradeoff): norm-quant with row-major (unswizzled) scales, the
standalone swizzle and unswizzle kernels, row shards gathered and swizzled
after the gather, and the bf16-output norm quantised after the gather.  All
bit-exact against the oracle."""

import numpy as np
import pytest
import torch

import mxfp8_norm_quant_gb300 as mx
import oracle as O
from mxfp8_norm_quant_gb300 import workloads as W
from mxtest import bf16_bits, np_u8

pytestmark = pytest.mark.gpu

# row counts that reach every row-ownership path of the dispatcher (rows
# split over 6 or 3 warps, one warp per row, the prefetching kernel; 720 and
# 800 rows sit on either side of the 3-warp kernel's one-round limit on a
# 152-SM GPU) with ragged 128-row blocks; widths with 1, 5 and 192 scale
# columns per row
SHAPES = [(1, 6144), (300, 6144), (720, 6144), (800, 6144), (1024, 6144), (5000, 6144), (77, 160), (640, 2048),
          (3000, 4096), (2500, 32), (9, 16384), (720, 6112), (800, 6112), (1024, 6112), (5000, 6112),
          (1000, 4160), (3000, 5184)]


def _ids(shapes):
    return [f"{m}x{h}" for m, h in shapes]


def _norm_rowmajor(x, w, eps, dev):
    M, H = x.shape
    q = torch.full((M, H), 0xA5, dtype=torch.uint8, device=dev)          # poison: every byte must be written
    s = torch.full((M * (H // 32),), 0xA5, dtype=torch.uint8, device=dev)
    mx.mx_rmsnorm_quant_ex(x.to(dev), w.to(dev), eps, q, s, M, H, mx.MX_SCALES_ROW_MAJOR)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    return np_u8(q), np_u8(s).reshape(M, H // 32)


@pytest.mark.parametrize("M,H", SHAPES, ids=_ids(SHAPES))
def test_rowmajor_scales(cuda_dev, M, H):
    x, w = W.norm_inputs(M, H, seed=M + 3 * H)
    rq, rs = O.mx_quantize_logical(O.gemma_rmsnorm_f32(bf16_bits(x), bf16_bits(w), 1e-6))
    gq, gs = _norm_rowmajor(x, w, 1e-6, cuda_dev)
    assert np.array_equal(gq, rq)
    assert np.array_equal(gs, rs)


def test_rowmajor_scales_unaligned_buffer(cuda_dev):
    # the row-major scale buffer needs no alignment: write it at byte offset 3
    M, H = 200, 2048
    x, w = W.norm_inputs(M, H, seed=8)
    q = torch.empty((M, H), dtype=torch.uint8, device=cuda_dev)
    buf = torch.full((M * (H // 32) + 16,), 0xA5, dtype=torch.uint8, device=cuda_dev)
    mx.mx_rmsnorm_quant_ex(x.to(cuda_dev), w.to(cuda_dev), 1e-6, q, buf.data_ptr() + 3, M, H,
                           mx.MX_SCALES_ROW_MAJOR)
    torch.cuda.synchronize()
    rq, rs = O.mx_quantize_logical(O.gemma_rmsnorm_f32(bf16_bits(x), bf16_bits(w), 1e-6))
    got = np_u8(buf)
    assert np.array_equal(np_u8(q), rq)
    assert np.array_equal(got[3:3 + M * (H // 32)].reshape(M, -1), rs)
    assert np.all(got[:3] == 0xA5) and np.all(got[3 + M * (H // 32):] == 0xA5)


@pytest.mark.parametrize("M,H", SHAPES + [(131072, 6144)], ids=_ids(SHAPES + [(131072, 6144)]))
def test_swizzle_kernels(cuda_dev, M, H):
    rng = np.random.default_rng(M + H)
    logical = rng.integers(0, 256, size=(M, H // 32), dtype=np.uint8)
    dev_in = torch.from_numpy(logical.reshape(-1).copy()).to(cuda_dev)
    sw = torch.full((mx.mx_scale_bytes(M, H),), 0xA5, dtype=torch.uint8, device=cuda_dev)
    mx.mx_swizzle_scales(dev_in, sw, M, H)
    back = torch.full((M * (H // 32),), 0xA5, dtype=torch.uint8, device=cuda_dev)
    mx.mx_unswizzle_scales(sw, back, M, H)
    torch.cuda.synchronize()
    assert np.array_equal(np_u8(sw), O.swizzle_scales(logical))
    assert np.array_equal(np_u8(back).reshape(M, -1), logical)


@pytest.mark.parametrize("shard_rows", [(512, 300), (1, 127, 129), (2000, 1500, 3)],
                         ids=["512+300", "1+127+129", "2000+1500+3"])
def test_gather_row_shards_then_swizzle(cuda_dev, shard_rows):
    # Sequence-parallel ranks normalise their own token rows with row-major
    # scales; the shards are concatenated by rows (the all-gather) and
    # swizzled once.  The result equals the fused norm of all rows and the
    # oracle, although the shards' 128-row blocks do not line up.
    H = 6144
    M = sum(shard_rows)
    x, w = W.norm_inputs(M, H, seed=21 + len(shard_rows))
    qs, ss, r0 = [], [], 0
    for n in shard_rows:
        q, s = _norm_rowmajor(x[r0:r0 + n], w, 1e-6, cuda_dev)
        qs.append(q)
        ss.append(s)
        r0 += n
    s_all = torch.from_numpy(np.concatenate(ss).reshape(-1).copy()).to(cuda_dev)
    sw = mx.swizzle_scales(s_all.view(M, H // 32), H)
    fq, fs = mx.rmsnorm_quant(x.to(cuda_dev), w.to(cuda_dev), 1e-6)
    torch.cuda.synchronize()
    assert np.array_equal(np.concatenate(qs), np_u8(fq))
    assert np.array_equal(np_u8(sw), np_u8(fs))
    rq, rs = O.rmsnorm_quant(bf16_bits(x), bf16_bits(w), 1e-6)
    assert np.array_equal(np_u8(sw), rs)
    assert np.array_equal(np.concatenate(qs), rq)


@pytest.mark.parametrize("M,H", SHAPES, ids=_ids(SHAPES))
def test_bf16_norm_then_quantise(cuda_dev, M, H):
    x, w = W.norm_inputs(M, H, seed=M + 5 * H)
    y = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device=cuda_dev)
    mx.mx_rmsnorm_bf16(x.to(cuda_dev), w.to(cuda_dev), 1e-6, y, M, H)
    torch.cuda.synchronize()
    ref = O.rmsnorm_bf16(bf16_bits(x), bf16_bits(w), 1e-6)
    assert np.array_equal(bf16_bits(y), ref)
    # quantise after the gather (here of one shard) with the plain quantiser
    gq, gs = mx.quant(y)
    torch.cuda.synchronize()
    rq, rs = O.quant(ref)
    assert np.array_equal(np_u8(gq), rq) and np.array_equal(np_u8(gs), rs)


@pytest.mark.parametrize("i", range(12))
def test_sp_forms_lane_block_boundaries(cuda_dev, i):
    # both sequence-parallel forms on either side of each kernel choice of the
    # lane-block dispatcher (the row counts of test_gpu_rowquant)
    from test_gpu_rowquant import lane_block_boundaries
    M = lane_block_boundaries(torch.cuda.get_device_properties(cuda_dev).multi_processor_count)[i]
    H = 6144
    x, w = W.norm_inputs(M, H, seed=M + 17)
    yf = O.gemma_rmsnorm_f32(bf16_bits(x), bf16_bits(w), 1e-6)
    rq, rs = O.mx_quantize_logical(yf)
    gq, gs = _norm_rowmajor(x, w, 1e-6, cuda_dev)
    assert np.array_equal(gq, rq) and np.array_equal(gs, rs)
    y = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device=cuda_dev)
    mx.mx_rmsnorm_bf16(x.to(cuda_dev), w.to(cuda_dev), 1e-6, y, M, H)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(y), O.f32_to_bf16_bits(yf))


@pytest.mark.parametrize("H", [6144, 1024, 3072, 8192, 16384, 6112])
def test_bf16_norm_degenerate_rows(cuda_dev, H):
    M = 64
    x, w = W.norm_inputs(M, H, seed=4)
    x = x.float()
    x[0] = 0.0
    x[1] = 1.0
    x[2] *= 1e15
    x[3] *= 1e-30
    x = x.to(torch.bfloat16)
    y = torch.empty((M, H), dtype=torch.bfloat16, device=cuda_dev)
    mx.mx_rmsnorm_bf16(x.to(cuda_dev), w.to(cuda_dev), 1e-6, y, M, H)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(y), O.rmsnorm_bf16(bf16_bits(x), bf16_bits(w), 1e-6))


def test_sp_forms_full_workload(cuda_dev):
    # the 32768 x 6144 norm in both sequence-parallel forms: every row against
    # the oracle (computed over row chunks), codes, row-major scales and bf16 y
    M, H = 32768, 6144
    x, w = W.norm_inputs(M, H, seed=77)
    xd, wd = x.to(cuda_dev), w.to(cuda_dev)
    q, s = mx.rmsnorm_quant_rowmajor(xd, wd, 1e-6)
    y = mx.rmsnorm_bf16(xd, wd, 1e-6)
    torch.cuda.synchronize()
    gq, gs, gy = np_u8(q), np_u8(s), bf16_bits(y)
    xb, wb = bf16_bits(x), bf16_bits(w)
    for r in range(0, M, 4096):
        yf = O.gemma_rmsnorm_f32(xb[r:r + 4096], wb, 1e-6)
        rq, rs = O.mx_quantize_logical(yf)
        assert np.array_equal(gq[r:r + 4096], rq), f"codes, rows {r}.."
        assert np.array_equal(gs[r:r + 4096], rs), f"row-major scales, rows {r}.."
        assert np.array_equal(gy[r:r + 4096], O.f32_to_bf16_bits(yf)), f"bf16 y, rows {r}.."
