"""Plain CPU oracle for the MXFP8 norm-quant + block-scaled GEMM path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, links or
runs this module; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may.  It shares no code with the CUDA path: no
helpers, tables or constants cross between the two.

What the pages fix and what is a reading
----------------------------------------
The vLLM pages (PR #64659 "Sequence parallelism and GEMM-RS for TP +
MegaMoE", PR #65496 "QuantizedActivation cannot be all-gathered under SP",
PR #64111 "MiniMax-M3.1-Flash model and kernels") name the pieces but print
no formula:

* a Gemma RMSNorm whose output is emitted directly as MXFP8
  (PR #65496, Overview and Details / Root cause: the norm output is a
  ``QuantizedActivation`` holding E4M3 data and UE8M0 scales);
* the scales in the ``F8_128x4`` swizzled layout the GEMM consumes
  (PR #64659, Details / "GEMM-RS with a quantized input"; PR #65496,
  Details / Tradeoff);
* an MXFP8 GEMM with N=6144, K=2048 (o_proj) and K=3072 (down_proj), BF16 out
  (PR #64659, GEMM-RS microbenchmark table).

Readings taken where the pages are silent:

R1  Gemma RMSNorm: y = x * rsqrt(mean(x^2) + eps) * (1 + w), mean over the
    whole row, eps inside the square root.
R2  Sum of squares in fp32, summed as a pairwise tree: the row is padded with
    +0.0 to the next power of two and sibling pairs are added level by level.
    (The quantised bytes must be reproducible bit for bit, so the order of
    the fp32 additions has to be part of the definition.)
R3  rsqrt is 1 / sqrt(v) with two correctly rounded fp32 operations; every
    other step is one correctly rounded fp32 operation, evaluated left to
    right: y = (x * r) * (1 + w).  y is not rounded to bf16 before quantising.
R4  MX scale: per 32 consecutive elements of a row, the shared exponent is
    E = floor(log2(amax)) - 8 (8 = largest exponent of E4M3), stored as the
    UE8M0 byte E + 127, clamped below at 0.  (The MX shared-exponent rule.)
R5  Element: t = y * 2^-E, then E4M3 (OCP "fn": bias 7, no infinities, max
    448) with round-to-nearest-even, magnitudes above 448 saturate to 448,
    the sign of zero kept.
R6  F8_128x4: the logical scale matrix S[R][C] (C = cols/32) is padded to
    Rp = ceil(R/128)*128 rows and Cp = ceil(C/4)*4 columns with zero bytes and
    stored in 512-byte blocks of 128 rows x 4 columns:
        off(r, c) = ((r//128) * (Cp//4) + c//4) * 512
                    + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4
R7  GEMM: C = A . B^T with A (M x K) and B (N x K) both K-contiguous; the
    oracle decodes both and multiplies in float64.
R8  The BF16 form of the norm (the sequence-parallel path of PR #65496, where
    the norm output stays BF16 through the all-gather and is quantised after
    it): the fp32 y of R1-R3 rounded to the nearest bf16, ties to even.

The floating-point steps that decide a quantised byte (R2-R5) run in fp32,
the precision the kernels use; the GEMM reference runs in float64.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "BLOCK",
    "bf16_bits_to_f32",
    "f32_to_bf16_bits",
    "e4m3_decode",
    "e4m3_encode",
    "ue8m0_decode",
    "scale_byte",
    "pairwise_sum_f32",
    "gemma_rmsnorm_f32",
    "mx_quantize_logical",
    "swizzle_offset",
    "swizzle_scales",
    "unswizzle_scales",
    "scale_bytes",
    "rmsnorm_quant",
    "rmsnorm_bf16",
    "quant",
    "mx_decode",
    "gemm_ref",
]

BLOCK = 32          # elements per UE8M0 scale (the "MX" block)
E4M3_EMAX = 8       # largest unbiased exponent of a finite E4M3 value (448 = 1.75 * 2^8)
E4M3_MAX = 448.0


# ---------------------------------------------------------------------------
# Element and scale formats
# ---------------------------------------------------------------------------

def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32, exactly (bf16 is the top half of fp32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even (R8).

    Dropping the low 16 bits of the fp32 pattern truncates; adding 0x7FFF plus
    the lowest kept bit first rounds to nearest with ties going to the even
    pattern (a carry out of the mantissa correctly bumps the exponent).
    Finite inputs only.
    """
    u = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    return ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """E4M3 ("fn" variant) byte -> float64.

    sign s = bit 7, exponent e = bits 6..3 (bias 7), mantissa m = bits 2..0.
    e > 0: (-1)^s (1 + m/8) 2^(e-7);  e == 0: (-1)^s (m/8) 2^-6;
    0x7F and 0xFF are NaN (the only NaN codes; there is no infinity).
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e > 0,
                   (1.0 + m / 8.0) * np.exp2(e - 7.0),
                   (m / 8.0) * np.exp2(-6.0))
    val = np.where(s == 1, -mag, mag)
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def e4m3_encode(t: np.ndarray) -> np.ndarray:
    """float32 -> E4M3 byte: round to nearest, ties to even, saturate at 448 (R5).

    Works on the exact float64 image of each fp32 input.  The grid spacing in
    the binade [2^e, 2^(e+1)) is 2^(e-3); below 2^-6 (subnormals) it is 2^-9.
    NaN inputs are outside the method's domain (finite inputs only).
    """
    t32 = np.asarray(t, dtype=np.float32)
    sign = ((t32.view(np.uint32) >> np.uint32(31)) & np.uint32(1)).astype(np.uint8)
    a = np.abs(t32.astype(np.float64))

    # exponent of the binade holding a: a = f * 2^ex with f in [0.5, 1)
    _, ex = np.frexp(a)
    e = np.maximum(ex.astype(np.int64) - 1, -6)          # subnormal binade uses 2^-6
    quantum = np.exp2((e - 3).astype(np.float64))
    v = np.rint(a / quantum) * quantum                    # np.rint: half to even
    v = np.where(a >= E4M3_MAX, E4M3_MAX, v)              # saturate (R5)
    v = np.minimum(v, E4M3_MAX)

    # encode the (exactly representable) value v
    _, vex = np.frexp(v)
    ve = vex.astype(np.int64) - 1
    normal = v >= np.exp2(-6.0)
    exp_field = np.where(normal, ve + 7, 0)
    mant = np.where(normal,
                    v / np.exp2(ve.astype(np.float64)) * 8.0 - 8.0,
                    v / np.exp2(-9.0))
    mant = mant.astype(np.int64)
    code = (sign.astype(np.int64) << 7) | (exp_field << 3) | mant
    return code.astype(np.uint8)


def ue8m0_decode(codes: np.ndarray) -> np.ndarray:
    """UE8M0 byte b -> 2^(b - 127) as float64; 0xFF is NaN."""
    b = np.asarray(codes, dtype=np.uint8).astype(np.float64)
    return np.where(b == 255, np.nan, np.exp2(b - 127.0))


def scale_byte(amax: np.ndarray) -> np.ndarray:
    """UE8M0 byte for a block whose largest magnitude is amax (fp32) (R4).

    floor(log2(amax)) is the unbiased exponent of amax, i.e. its biased
    exponent field minus 127, for normal amax.  Subtracting E4M3's emax (8)
    and re-biasing gives byte = field - 8, clamped at 0 (zero or tiny blocks).
    """
    a = np.asarray(amax, dtype=np.float32)
    field = ((a.view(np.uint32) >> np.uint32(23)) & np.uint32(0xFF)).astype(np.int64)
    return np.maximum(field - E4M3_EMAX, 0).astype(np.uint8)


# ---------------------------------------------------------------------------
# Gemma RMSNorm in fp32 (R1-R3)
# ---------------------------------------------------------------------------

def pairwise_sum_f32(v: np.ndarray) -> np.ndarray:
    """Row sums of a 2-D float32 array by the pairwise tree of R2."""
    v = np.asarray(v, dtype=np.float32)
    rows, n = v.shape
    width = 1
    while width < n:
        width *= 2
    level = np.zeros((rows, width), dtype=np.float32)
    level[:, :n] = v
    while level.shape[1] > 1:
        level = level[:, 0::2] + level[:, 1::2]       # fp32 + fp32 -> fp32, RNE
    return level[:, 0]


def gemma_rmsnorm_f32(x_bits: np.ndarray, w_bits: np.ndarray, eps: float) -> np.ndarray:
    """y = x * rsqrt(mean(x^2) + eps) * (1 + w), all in fp32 (R1-R3).

    x_bits: (M, H) uint16 bf16 patterns; w_bits: (H,) uint16; eps as fp32.
    """
    xf = bf16_bits_to_f32(x_bits)
    wf = bf16_bits_to_f32(w_bits)
    h = xf.shape[1]
    with np.errstate(over="ignore"):               # a square past the fp32 range is +inf, as on the GPU
        sq = xf * xf                               # fp32 products
        ss = pairwise_sum_f32(sq)                  # (M,)
    ms = ss / np.float32(h)                        # mean
    v = ms + np.float32(eps)
    s = np.sqrt(v)                                 # correctly rounded fp32 sqrt
    r = np.float32(1.0) / s                        # correctly rounded fp32 divide
    g = np.float32(1.0) + wf                       # Gemma gain (1 + w)
    y = (xf * r[:, None]) * g[None, :]
    assert y.dtype == np.float32
    return y


# ---------------------------------------------------------------------------
# MX quantisation (R4, R5) and the F8_128x4 layout (R6)
# ---------------------------------------------------------------------------

def mx_quantize_logical(y: np.ndarray):
    """fp32 (R, C) -> (E4M3 codes (R, C) uint8, logical scales (R, C/32) uint8)."""
    y = np.asarray(y, dtype=np.float32)
    rows, cols = y.shape
    assert cols % BLOCK == 0
    blocks = y.reshape(rows, cols // BLOCK, BLOCK)
    amax = np.max(np.abs(blocks), axis=2)                          # fp32
    sb = scale_byte(amax)                                          # (R, C/32)
    # 2^-E = 2^(127 - byte): a normal fp32 power of two for byte in [0, 246]
    inv = np.exp2(127.0 - sb.astype(np.float64)).astype(np.float32)
    t = blocks * inv[:, :, None]                                   # fp32 multiply
    q = e4m3_encode(t).reshape(rows, cols)
    return q, sb


def scale_bytes(rows: int, cols: int) -> int:
    """Size in bytes of the swizzled scale buffer for a rows x cols operand."""
    c = cols // BLOCK
    return (-(-rows // 128) * 128) * (-(-c // 4) * 4)


def swizzle_offset(r, c, cols_scale: int):
    """Byte offset of logical scale (r, c) in the F8_128x4 layout (R6).

    cols_scale is C, the number of logical scale columns (cols / 32).
    """
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    cp4 = -(-cols_scale // 4)                                  # Cp / 4
    return ((r // 128) * cp4 + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4


def swizzle_scales(s: np.ndarray) -> np.ndarray:
    """Logical (R, C) scale bytes -> flat swizzled buffer, padding bytes zero."""
    s = np.asarray(s, dtype=np.uint8)
    rows, c = s.shape
    rp = -(-rows // 128) * 128
    cp = -(-c // 4) * 4
    out = np.zeros(rp * cp, dtype=np.uint8)
    rr, cc = np.meshgrid(np.arange(rows), np.arange(c), indexing="ij")
    out[swizzle_offset(rr, cc, c)] = s
    return out


def unswizzle_scales(buf: np.ndarray, rows: int, c: int) -> np.ndarray:
    """Flat swizzled buffer -> logical (rows, c) scale bytes."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    rr, cc = np.meshgrid(np.arange(rows), np.arange(c), indexing="ij")
    return buf[swizzle_offset(rr, cc, c)]


# ---------------------------------------------------------------------------
# The two quantising operations and the GEMM reference
# ---------------------------------------------------------------------------

def rmsnorm_quant(x_bits: np.ndarray, w_bits: np.ndarray, eps: float):
    """Fused Gemma RMSNorm + MXFP8 quantisation of an (M, H) bf16 input.

    Returns (q: (M, H) uint8 E4M3 codes, s: flat swizzled UE8M0 scales).
    """
    y = gemma_rmsnorm_f32(x_bits, w_bits, eps)
    q, sb = mx_quantize_logical(y)
    return q, swizzle_scales(sb)


def rmsnorm_bf16(x_bits: np.ndarray, w_bits: np.ndarray, eps: float) -> np.ndarray:
    """The Gemma RMSNorm alone, rounded to bf16 (R8).  Returns (M, H) uint16
    bit patterns."""
    return f32_to_bf16_bits(gemma_rmsnorm_f32(x_bits, w_bits, eps))


def quant(x_bits: np.ndarray):
    """Plain MXFP8 quantisation of an (R, C) bf16 operand (the GEMM inputs)."""
    q, sb = mx_quantize_logical(bf16_bits_to_f32(x_bits))
    return q, swizzle_scales(sb)


def mx_decode(q: np.ndarray, s_swizzled: np.ndarray) -> np.ndarray:
    """Decode an MXFP8 operand (codes + swizzled scales) to float64 (R, C)."""
    q = np.asarray(q, dtype=np.uint8)
    rows, cols = q.shape
    c = cols // BLOCK
    sb = unswizzle_scales(s_swizzled, rows, c)
    scale = ue8m0_decode(sb)                                        # (R, C/32)
    return (e4m3_decode(q).reshape(rows, c, BLOCK) * scale[:, :, None]).reshape(rows, cols)


def gemm_ref(a_q, a_s, b_q, b_s) -> np.ndarray:
    """float64 reference of C = dec(A) . dec(B)^T (R7).

    a_q: (M, K) codes, a_s: swizzled A scales; b_q: (N, K), b_s likewise.
    """
    return mx_decode(a_q, a_s) @ mx_decode(b_q, b_s).T
