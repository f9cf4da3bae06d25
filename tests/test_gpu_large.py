"""GPU parity at the largest sizes the C ABI takes: tensors past 2^32 bytes
(64-bit addressing in every kernel) and GEMM dimensions at their 2^20 limit.

The inputs are built on the device from a seeded block of rows: copy j of
the block is scaled by 2^((j % 16) - 8), exact in bf16, so rows are distinct
and every row's bytes are known.  The oracle runs on sampled rows (the first,
the last, both sides of every block and 2^31-byte boundary, and seeded
random ones), read back from the device."""

import numpy as np
import pytest
import torch

import mxfp8_norm_quant_gb300 as mx
import oracle as O
from mxfp8_norm_quant_gb300 import workloads as W
from mxtest import bf16_bits, gemm_close, np_u8

pytestmark = pytest.mark.gpu


def _tiled(block: torch.Tensor, copies: int, dev) -> torch.Tensor:
    """copies x block rows on the device; copy j = block * 2^((j % 16) - 8)."""
    b = block.to(dev)
    r = b.shape[0]
    out = torch.empty((copies * r, b.shape[1]), dtype=torch.bfloat16, device=dev)
    for j in range(copies):
        out[j * r:(j + 1) * r] = b * (2.0 ** ((j % 16) - 8))
    return out


def _sample_rows(m: int, row_bytes: int, seed: int) -> np.ndarray:
    rows = {0, 1, 127, 128, m // 2 - 1, m // 2, m - 129, m - 128, m - 2, m - 1}
    # both sides of every 2^31-byte boundary of the input
    for t in range(1, ((m * row_bytes) >> 31) + 1):
        r = (t << 31) // row_bytes
        rows.update(v for v in (r - 1, r, r + 1) if 0 <= v < m)
    rows.update(np.random.default_rng(seed).integers(0, m, 16).tolist())
    return np.array(sorted(v for v in rows if 0 <= v < m), dtype=np.int64)


def _scales_at(buf: np.ndarray, rows: np.ndarray, c: int) -> np.ndarray:
    """Logical (row, column) scale bytes of `rows` from an F8_128x4 buffer."""
    rr, cc = np.meshgrid(rows, np.arange(c), indexing="ij")
    return buf[O.swizzle_offset(rr, cc, c)]


def test_norm_and_quant_past_4gb(cuda_dev):
    # 262144 x 16384 bf16: x is 8 GiB, the codes 4 GiB
    M, H = 1 << 18, 16384
    block, w = W.norm_inputs(1024, H, seed=21, outlier_frac=0.01, zero_block_frac=1 / 128)
    x = _tiled(block, M // 1024, cuda_dev)
    wd = w.to(cuda_dev)
    q = torch.empty((M, H), dtype=torch.uint8, device=cuda_dev)
    s = torch.empty(mx.mx_scale_bytes(M, H), dtype=torch.uint8, device=cuda_dev)
    mx.mx_rmsnorm_quant(x, wd, 1e-6, q, s, M, H)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    rows = _sample_rows(M, 2 * H, seed=1)
    idx = torch.from_numpy(rows).to(cuda_dev)
    xb = bf16_bits(x[idx])
    rq, rs = O.mx_quantize_logical(O.gemma_rmsnorm_f32(xb, bf16_bits(w), 1e-6))
    assert np.array_equal(np_u8(q[idx]), rq)
    assert np.array_equal(_scales_at(np_u8(s), rows, H // 32), rs)
    del q, s
    # the plain quantiser over the same 8 GiB operand
    q2 = torch.empty((M, H), dtype=torch.uint8, device=cuda_dev)
    s2 = torch.empty(mx.mx_scale_bytes(M, H), dtype=torch.uint8, device=cuda_dev)
    mx.mx_quant_weights(x, q2, s2, M, H)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    rq2, rs2 = O.mx_quantize_logical(O.bf16_bits_to_f32(xb))
    assert np.array_equal(np_u8(q2[idx]), rq2)
    assert np.array_equal(_scales_at(np_u8(s2), rows, H // 32), rs2)
    del x, q2, s2
    torch.cuda.empty_cache()


def _pm1_operand(rows, cols, seed, dev):
    """Seeded MXFP8 operand of any width (the quantiser takes rows of at most
    16384) whose GEMM is exact in fp32: E4M3 codes of +1, -1 and 0 (0x38,
    0xB8, 0x00) and every scale byte 127 (2^0), so every dot product is an
    integer of magnitude at most K and exact in fp32."""
    g = torch.Generator().manual_seed(seed)
    pick = torch.randint(0, 3, (rows, cols), dtype=torch.uint8, generator=g)
    codes = torch.tensor([0x38, 0xB8, 0x00], dtype=torch.uint8)
    q = codes[pick.long()]
    s = torch.full((mx.mx_scale_bytes(rows, cols),), 127, dtype=torch.uint8)
    return q.to(dev), s.to(dev)


def _gemm_check(cuda_dev, M, N, K, seed, quant_out):
    if K <= 16384:
        a_blk, wt = W.gemm_operands(min(M, 4096), K, seed=seed, n=N)
        a = _tiled(a_blk, M // a_blk.shape[0], cuda_dev)
        aq = torch.empty((M, K), dtype=torch.uint8, device=cuda_dev)
        as_ = torch.empty(mx.mx_scale_bytes(M, K), dtype=torch.uint8, device=cuda_dev)
        mx.mx_quant_weights(a, aq, as_, M, K)
        del a
        bq, bs_ = mx.quant(wt.to(cuda_dev))
    else:
        aq, as_ = _pm1_operand(M, K, seed, cuda_dev)
        bq, bs_ = _pm1_operand(N, K, seed + 1000, cuda_dev)
    c = torch.empty((M, N), dtype=torch.bfloat16, device=cuda_dev)
    mx.mx_gemm(aq, as_, bq, bs_, c, M, N, K)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    rows = _sample_rows(M, K, seed=seed)
    idx = torch.from_numpy(rows).to(cuda_dev)
    a_rows = O.swizzle_scales(_scales_at(np_u8(as_), rows, K // 32))
    ref = O.gemm_ref(np_u8(aq[idx]), a_rows, np_u8(bq), np_u8(bs_))
    if K > 16384:
        # integer dot products: C is their bf16 rounding, bit for bit
        assert np.array_equal(bf16_bits(c[idx]), O.f32_to_bf16_bits(ref.astype(np.float32)))
    else:
        ok, worst = gemm_close(c[idx], ref)
        assert ok, f"worst err/tol = {worst:.3f}"
    if quant_out:
        # the MXFP8-output epilogue equals the quantisation of the bf16 C of
        # the same tile: the oracle's on the sampled rows, and the library
        # quantiser's over the whole output where C's rows fit it
        cq = torch.empty((M, N), dtype=torch.uint8, device=cuda_dev)
        cs = torch.empty(mx.mx_scale_bytes(M, N), dtype=torch.uint8, device=cuda_dev)
        mx.mx_gemm_quant(aq, as_, bq, bs_, cq, cs, M, N, K)
        torch.cuda.synchronize()
        assert mx.mx_device_fault() == 0
        oq, os_ = O.mx_quantize_logical(O.bf16_bits_to_f32(bf16_bits(c[idx])))
        assert np.array_equal(np_u8(cq[idx]), oq)
        assert np.array_equal(_scales_at(np_u8(cs), rows, N // 32), os_)
        if N <= 16384:
            rq, rs = mx.quant(c)
            torch.cuda.synchronize()
            assert torch.equal(cq, rq) and torch.equal(cs, rs)


def test_gemm_max_m_past_4gb(cuda_dev):
    # M = 2^20 (the limit), K = 4096: A is 4 GiB of codes, C 4 GiB of bf16
    _gemm_check(cuda_dev, 1 << 20, 2048, 4096, seed=31, quant_out=True)
    torch.cuda.empty_cache()


def test_gemm_max_k(cuda_dev):
    # K = 2^20 (the limit): 8192 K steps of 128 through one tile of pairs, on
    # operands whose GEMM is exact (a K step missed or repeated changes the
    # integer result).  Uniformly random codes are not used here: their sums
    # over 2^20 products cancel so far that the elementwise 1e-2 relative bound
    # fails near zero, by the accumulation's rounding, identically for every tile
    _gemm_check(cuda_dev, 256, 128, 1 << 20, seed=32, quant_out=False)
    torch.cuda.empty_cache()


def test_gemm_max_n(cuda_dev):
    # N = 2^20 (the limit): 16384 tiles of 128 x 64 over one tile row of A
    _gemm_check(cuda_dev, 128, 1 << 20, 64, seed=33, quant_out=True)
    torch.cuda.empty_cache()
