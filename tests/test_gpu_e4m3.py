"""Exhaustive check of the kernels' fp32 -> E4M3 conversion (round to nearest
even, saturation at 448) against the oracle over all 2^32 fp32 bit patterns
(NaN inputs excluded: they are outside the method's domain).

The oracle's encoder is a monotone step function of |t|; its 126 step
positions are found with the oracle itself (binary search), and expanded on
the device with searchsorted.  A CPU test checks that this expansion equals
the oracle on random patterns."""

import numpy as np
import pytest
import torch

import mxfp8_norm_quant_gb300 as mx
import oracle as O
from mxtest import e4m3_thresholds

pytestmark = pytest.mark.gpu


def test_e4m3_all_fp32_patterns(cuda_dev):
    thr = torch.from_numpy(e4m3_thresholds(O.e4m3_encode)).to(cuda_dev)
    chunk = 1 << 28
    out = torch.empty(chunk, dtype=torch.uint8, device=cuda_dev)
    mismatches = 0
    first = None
    for start in range(0, 1 << 32, chunk):
        bits = torch.arange(start, start + chunk, dtype=torch.int64, device=cuda_dev)
        inp = bits.to(torch.int32).view(torch.float32)          # wraps to the same 32-bit patterns
        mx.mx_e4m3_encode_f32(inp, out, chunk)
        mag = bits & 0x7FFFFFFF
        sign = (bits >> 31) & 1
        expect = (torch.searchsorted(thr, mag, right=True) | (sign << 7)).to(torch.uint8)
        nan = mag > 0x7F800000
        bad = (out != expect) & ~nan
        n = int(bad.sum())
        if n and first is None:
            idx = int(torch.nonzero(bad)[0])
            first = (hex(start + idx), int(out[idx]), int(expect[idx]))
        mismatches += n
        del bits, inp, mag, sign, expect, nan, bad
    torch.cuda.synchronize()
    assert mismatches == 0, f"{mismatches} mismatches; first (pattern, got, expected) = {first}"


def test_e4m3_probe_examples(cuda_dev):
    vals = np.float32([0.0, -0.0, 1.0, 448.0, 464.0, 480.0, 1e9, -1e9, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10,
                       np.inf, -np.inf, 272.0, 304.0, 12.8])
    inp = torch.from_numpy(vals).to(cuda_dev)
    out = torch.empty(len(vals), dtype=torch.uint8, device=cuda_dev)
    mx.mx_e4m3_encode_f32(inp, out, len(vals))
    torch.cuda.synchronize()
    assert out.cpu().numpy().tolist() == O.e4m3_encode(vals).tolist()
