"""Shared helpers for the parity tests: moving seeded inputs between torch and
the oracle's numpy arrays, and the GEMM tolerance."""

import numpy as np
import torch

# |gpu - ref| <= GEMM_RTOL * (|ref| + 1): bf16 output rounding (2^-9 relative)
# plus fp32 accumulation, with a wide margin.
GEMM_RTOL = 1e-2


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> uint16 numpy bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def np_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def to_dev(a, dev) -> torch.Tensor:
    if isinstance(a, np.ndarray):
        a = torch.from_numpy(np.ascontiguousarray(a))
    return a.to(dev).contiguous()


def gemm_close(got_bf16: torch.Tensor, ref: np.ndarray):
    """(ok, worst ratio) for the element-wise tolerance test."""
    g = got_bf16.detach().float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    lim = GEMM_RTOL * (np.abs(ref) + 1.0)
    ratio = float(np.max(err / lim)) if err.size else 0.0
    return bool(np.all(err <= lim)) and bool(np.all(np.isfinite(g))), ratio


def e4m3_thresholds(encode) -> np.ndarray:
    """For the oracle's encoder (monotone in |t|), the smallest non-negative
    fp32 bit pattern that encodes to each code 1..126, by binary search."""
    codes = np.arange(1, 127, dtype=np.int64)
    lo = np.zeros(codes.shape, dtype=np.int64)            # encode(lo) < code
    hi = np.full(codes.shape, 0x7F800000, dtype=np.int64)  # encode(hi) >= code (+inf saturates)
    while np.any(hi - lo > 1):
        mid = (lo + hi) // 2
        c = encode(mid.astype(np.uint32).view(np.float32)).astype(np.int64)
        ge = c >= codes
        hi = np.where(ge, mid, hi)
        lo = np.where(ge, lo, mid)
    return hi
