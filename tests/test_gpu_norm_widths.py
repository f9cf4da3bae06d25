"""GPU parity of the norm at widths other than the models' 6144: every kernel
choice the lane-block dispatcher makes for rows of 64..4096 and 6145..16384
elements (H % 64 == 0), in all three output forms (E4M3 codes with swizzled
or row-major scales, and the BF16 rows), bit for bit against the oracle.

The row counts sit on either side of the dispatcher's rows-per-SM limits for
this GPU's SM count, and the widths have a whole or a partial last
1024-element chunk (a partial chunk leaves lanes, and with several warps per
row whole warps, without elements)."""

import numpy as np
import pytest
import torch

import mxfp8_norm_quant_gb300 as mx
import oracle as O
from mxfp8_norm_quant_gb300 import workloads as W
from mxtest import bf16_bits, np_u8

pytestmark = pytest.mark.gpu

ALL = ("swizzled", "rowmajor", "bf16")


def width_cases(s):
    """(H, M, forms) for a GPU of s SMs; the comment of each group names the
    kernels (<warps per row, chunks per warp, rows per CTA>) it reaches."""
    return [
        # H <= 512: chunked kernels up to 16 rows per SM, then <1,1,32>;
        # 513..1024: <1,1,8> to 8 rows per SM, <1,1,16> to 16, <1,1,32>
        (512, 16 * s, ALL), (512, 16 * s + 1, ALL), (64, 16 * s + 1, ALL), (576, 100, ALL),
        (1024, 8 * s, ALL), (1024, 8 * s + 1, ALL), (960, 16 * s + 1, ALL),
        # 1025..2048: <2,1,4> to 4 rows per SM, <2,1,8> to 8, <1,2,16> to 64, <1,2,24>
        (1088, 5, ALL), (1536, 4 * s, ALL), (2048, 4 * s + 1, ALL), (1536, 8 * s + 1, ALL),
        (2048, 64 * s, ALL), (1536, 64 * s + 1, ALL),
        # 2049..3072: <3,1,2> to 2 rows per SM, <3,1,4> to 4, <3,1,8> to 8, <1,4,16>
        (3072, 1, ALL), (2112, 2 * s, ALL), (2560, 2 * s + 1, ALL), (3072, 8 * s, ALL), (2112, 8 * s + 1, ALL),
        (3072, 5000, ALL),
        # 3073..4096: <4,1,2> to 2 rows per SM, <4,1,4> to 4, <2,2,8> to 16, <1,4,12>
        (4096, 3, ALL), (3136, 2 * s + 1, ALL), (4096, 4 * s + 1, ALL), (3136, 16 * s, ALL),
        (4096, 16 * s + 1, ALL), (3136, 6000, ALL),
        # 6145..8192: <8,1,2> to 1.5 rows per SM, <4,2,4> to 16 (BF16 form: to
        # 64, then <4,2,3>), <4,2,6>
        (8192, 1, ALL), (7168, 3 * s // 2, ALL), (7168, 3 * s // 2 + 1, ALL), (6208, 16 * s + 1, ALL),
        (8192, 3000, ALL), (6208, 64 * s + 1, ("bf16",)),
        # 8193..16384: <8,2,2> to 4 rows per SM, then <4,4,3> to 12288 elements
        # and <8,2,3> beyond (BF16 form: <8,2,3>, and <8,2,2> past 9216
        # elements and 64 rows per SM)
        (16384, 5, ALL), (8256, 4 * s, ALL), (8256, 4 * s + 1, ALL), (12288, 3000, ALL), (12352, 700, ALL),
        (16384, 1000, ALL), (9280, 64 * s + 1, ("bf16",)),
    ]


N_CASES = len(width_cases(152))


def _run(form, xd, wd, M, H, dev):
    if form == "bf16":
        y = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device=dev)
        mx.mx_rmsnorm_bf16(xd, wd, 1e-6, y, M, H)
        torch.cuda.synchronize()
        return bf16_bits(y)
    q = torch.full((M, H), 0xA5, dtype=torch.uint8, device=dev)        # poison: every byte must be written
    if form == "swizzled":
        s = torch.full((mx.mx_scale_bytes(M, H),), 0xA5, dtype=torch.uint8, device=dev)
        mx.mx_rmsnorm_quant(xd, wd, 1e-6, q, s, M, H)
    else:
        s = torch.full((M * (H // 32),), 0xA5, dtype=torch.uint8, device=dev)
        mx.mx_rmsnorm_quant_ex(xd, wd, 1e-6, q, s, M, H, mx.MX_SCALES_ROW_MAJOR)
    torch.cuda.synchronize()
    return np_u8(q), np_u8(s)


@pytest.mark.parametrize("i", range(N_CASES))
def test_norm_other_widths(cuda_dev, i):
    H, M, forms = width_cases(torch.cuda.get_device_properties(cuda_dev).multi_processor_count)[i]
    x, w = W.norm_inputs(M, H, seed=H * 31 + M, outlier_frac=0.01, zero_block_frac=1 / 128)
    xd, wd = x.to(cuda_dev), w.to(cuda_dev)
    yf = O.gemma_rmsnorm_f32(bf16_bits(x), bf16_bits(w), 1e-6)
    if "bf16" in forms:
        assert np.array_equal(_run("bf16", xd, wd, M, H, cuda_dev), O.f32_to_bf16_bits(yf)), "bf16 rows"
    if "swizzled" in forms or "rowmajor" in forms:
        rq, rs = O.mx_quantize_logical(yf)
        del yf
        for form in ("swizzled", "rowmajor"):
            gq, gs = _run(form, xd, wd, M, H, cuda_dev)
            bad = np.argwhere(gq != rq)
            assert bad.size == 0, f"{form}: {len(bad)} code mismatches, first at {bad[:5].tolist()}"
            want = O.swizzle_scales(rs) if form == "swizzled" else rs.reshape(-1)
            bad_s = np.flatnonzero(gs != want)
            assert bad_s.size == 0, f"{form}: {bad_s.size} scale-byte mismatches, first {bad_s[:8].tolist()}"
    assert mx.mx_device_fault() == 0
