"""GPU parity of mx_gemm_quant, the GEMM whose output leaves as an MXFP8
operand (E4M3 codes + F8_128x4 UE8M0 scales of C rounded to bf16).

* Exact: operands whose products and partial sums are exact in fp32 make C,
  its bf16 rounding and hence every code and scale byte a function of the
  oracle alone: the oracle's quantiser applied to the oracle's GEMM must
  match bit for bit, padding included.
* Random operands: the decoded output is within the GEMM tolerance plus the
  MXFP8 quantisation error of the oracle's float64 C; codes and scale bytes
  equal the oracle's except where C lies within rounding distance of a
  decision boundary (rare, and then off by one step only).
* Consistency of two CUDA paths: for one tile, the epilogue's bytes equal
  mx_quant_weights applied to mx_gemm_ex's bf16 output, bit for bit.
"""

import numpy as np
import pytest
import torch

import mxfp8_norm_quant_gb300 as mx
import oracle as O
from mxfp8_norm_quant_gb300 import workloads as W
from mxtest import GEMM_RTOL, bf16_bits, np_u8, to_dev

pytestmark = pytest.mark.gpu

TILES = [(128, 64), (128, 128), (128, 192), (256, 128), (256, 192), (256, 256)]
TILE_IDS = [f"{m}x{n}" for m, n in TILES]


def _gemm_quant(aq, as_, bq, bs, M, N, K, dev, tile=(0, 0)):
    q = torch.full((M, N), 0xA5, dtype=torch.uint8, device=dev)          # poison: every byte must be written
    s = torch.full((mx.mx_scale_bytes(M, N),), 0xA5, dtype=torch.uint8, device=dev)
    mx.mx_gemm_quant(to_dev(aq, dev), to_dev(as_, dev), to_dev(bq, dev), to_dev(bs, dev), q, s, M, N, K, *tile)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    return np_u8(q), np_u8(s)


def _oracle_quantised(ref):
    """The oracle's MXFP8 form of a float64 C: fp32, bf16 (RNE), then quant."""
    return O.quant(O.f32_to_bf16_bits(ref.astype(np.float32)))


@pytest.mark.parametrize("M,N,K", [(384, 320, 640), (300, 160, 256), (1, 96, 32), (129, 6144, 512)])
@pytest.mark.parametrize("tile", TILES, ids=TILE_IDS)
def test_exact_against_oracle(cuda_dev, M, N, K, tile):
    # entries in {-1, 0, 1} with scales x1/x2 on A and x0.5/x1 on B:
    # |partial sums| <= 2K <= 1280 at a granularity of 0.5 (12 significant
    # bits), exact in any order, even in an accumulator narrower than fp32
    rng = np.random.default_rng(M * 7 + N + K + tile[1])
    ai = rng.integers(-1, 2, size=(M, K))
    bi = rng.integers(-1, 2, size=(N, K))
    aq = O.e4m3_encode(ai.astype(np.float32))
    bq = O.e4m3_encode(bi.astype(np.float32))
    asb = O.swizzle_scales(rng.integers(127, 129, size=(M, K // 32), dtype=np.uint8))
    bsb = O.swizzle_scales(rng.integers(126, 128, size=(N, K // 32), dtype=np.uint8))
    ref = O.gemm_ref(aq, asb, bq, bsb)
    assert np.all(ref.astype(np.float32).astype(np.float64) == ref)      # C is exact in fp32
    rq, rs = _oracle_quantised(ref)
    gq, gs = _gemm_quant(aq, asb, bq, bsb, M, N, K, cuda_dev, tile)
    bad = np.argwhere(gq != rq)
    assert bad.size == 0, f"{len(bad)} code mismatches, first {bad[:4].tolist()}"
    assert np.array_equal(gs, rs)


def _check_against_float64(gq, gs, ref):
    """Decoded output vs the float64 C within the GEMM tolerance plus the
    quantisation error at the output's own block scale; codes and scale bytes
    vs the oracle's own quantisation of C."""
    M, N = ref.shape
    dec = O.mx_decode(gq, gs)
    sb = O.unswizzle_scales(gs, M, N // 32).astype(np.float64)
    e = np.repeat(np.exp2(sb - 127.0), 32, axis=1)                 # 2^E of each element's block
    a = np.abs(ref)
    quant_err = np.maximum(a * 2.0 ** -4, e * 2.0 ** -10) + np.maximum(0.0, a - 448.0 * e)
    lim = GEMM_RTOL * (a + 1.0) + quant_err
    err = np.abs(dec - ref)
    assert np.all(np.isfinite(dec))
    assert np.all(err <= lim), f"worst err/lim = {float(np.max(err / lim)):.3f}"
    rq, rs = _oracle_quantised(ref)
    rsb = O.unswizzle_scales(rs, M, N // 32).astype(np.int64)
    assert np.max(np.abs(rsb - sb.astype(np.int64))) <= 1
    assert np.mean(rsb == sb) >= 0.999
    assert np.mean(gq == rq) >= 0.99


SHAPES = [(128, 6144, 2048), (300, 416, 288), (129, 256, 4096), (512, 1024, 3072), (77, 160, 160)]


@pytest.mark.parametrize("M,N,K", SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in SHAPES])
@pytest.mark.parametrize("tile", [(0, 0)] + TILES, ids=["auto"] + TILE_IDS)
def test_random_against_oracle(cuda_dev, M, N, K, tile):
    a, wt = W.gemm_operands(M, K, seed=M + N + K, n=N)
    aq, as_ = O.quant(bf16_bits(a))
    bq, bs_ = O.quant(bf16_bits(wt))
    ref = O.gemm_ref(aq, as_, bq, bs_)
    gq, gs = _gemm_quant(aq, as_, bq, bs_, M, N, K, cuda_dev, tile)
    # padding of the scale buffer (rows past M, scale columns past N/32) is zero
    full = gs.reshape(-1)
    logical = np.zeros(full.shape, dtype=bool)
    rr, cc = np.meshgrid(np.arange(M), np.arange(N // 32), indexing="ij")
    logical[O.swizzle_offset(rr, cc, N // 32)] = True
    assert np.all(full[~logical] == 0)
    _check_against_float64(gq, gs, ref)


@pytest.mark.parametrize("M,N,K", [(300, 448, 256), (1000, 6144, 2048), (77, 160, 96)])
@pytest.mark.parametrize("tile", TILES, ids=TILE_IDS)
def test_epilogue_equals_quantised_bf16_gemm(cuda_dev, M, N, K, tile):
    # two CUDA paths with the same accumulators: the fused epilogue and the
    # plain quantiser run on the bf16 GEMM of the same tile
    a, wt = W.gemm_operands(M, K, seed=3 * M + K, n=N)
    aq, as_ = mx.quant(a.to(cuda_dev))
    bq, bs_ = mx.quant(wt.to(cuda_dev))
    c = torch.empty((M, N), dtype=torch.bfloat16, device=cuda_dev)
    mx.mx_gemm_ex(aq, as_, bq, bs_, c, M, N, K, *tile)
    cq, cs = mx.quant(c)
    gq, gs = _gemm_quant(aq, as_, bq, bs_, M, N, K, cuda_dev, tile)
    assert np.array_equal(gq, np_u8(cq))
    assert np.array_equal(gs, np_u8(cs))


def test_codes_16_byte_aligned_only(cuda_dev):
    # a code buffer 16- but not 32-byte aligned takes the 16-byte store path
    M, N, K = 256, 448, 256
    a, wt = W.gemm_operands(M, K, seed=9, n=N)
    aq, as_ = O.quant(bf16_bits(a))
    bq, bs_ = O.quant(bf16_bits(wt))
    big = torch.full((M * N + 32,), 0xA5, dtype=torch.uint8, device=cuda_dev)
    off = 16 if big.data_ptr() % 32 == 0 else 0
    q = big[off:off + M * N].view(M, N)
    assert q.data_ptr() % 32 == 16
    s = torch.empty(mx.mx_scale_bytes(M, N), dtype=torch.uint8, device=cuda_dev)
    mx.mx_gemm_quant(to_dev(aq, cuda_dev), to_dev(as_, cuda_dev), to_dev(bq, cuda_dev), to_dev(bs_, cuda_dev), q, s,
                     M, N, K, 128, 192)
    torch.cuda.synchronize()
    _check_against_float64(np_u8(q), np_u8(s), O.gemm_ref(aq, as_, bq, bs_))


@pytest.mark.parametrize("name,k", [("m1024", 3072), ("m4096_rowscale", 2048), ("m32768_stress", 3072)])
def test_workload_full_size_every_row(cuda_dev, name, k):
    # the full-size MXFP8-output GEMM, every row against the float64 oracle;
    # the oracle runs over row chunks of 4096 (a multiple of 128, so each
    # chunk's swizzled scales are one contiguous span of the full buffer)
    wl = W.WORKLOADS[name]
    a, wt = wl.gemm(k, 0)
    M, N = a.shape[0], wt.shape[0]
    aq, as_ = mx.quant(a.to(cuda_dev))
    bq, bs_ = mx.quant(wt.to(cuda_dev))
    q, s = mx.gemm_quant(aq, as_, bq, bs_)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    gq, gs = np_u8(q), np_u8(s)
    bq_o, bs_o = O.quant(bf16_bits(wt))
    ab = bf16_bits(a)
    span = O.scale_bytes(4096, N)
    for r in range(0, M, 4096):
        rows = min(4096, M - r)
        aq_o, as_o = O.quant(ab[r:r + rows])
        ref = O.gemm_ref(aq_o, as_o, bq_o, bs_o)
        _check_against_float64(gq[r:r + rows], gs[r // 4096 * span:r // 4096 * span + O.scale_bytes(rows, N)], ref)
