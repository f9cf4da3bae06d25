"""Pins for the CPU oracle, checked against things other than the oracle itself.

Each test ties one part of the oracle to a hand-worked value, a closed form, a
format invariant, an independent library decoder, or brute force, so that a
plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a wrong rounding rule) fails at least one of them.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mx_blocks.txt")

# all non-negative finite E4M3 values, indexed by code, straight from the
# format's bit-field definition (written out here independently of the oracle)
def _e4m3_table():
    vals = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        v = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        vals.append(float(v))
    return np.array(vals, dtype=np.float64)


E4M3_POS = _e4m3_table()


def _brute_e4m3(t32):
    """Nearest finite E4M3 by exhaustive search; ties go to the even code; >448 -> 448."""
    t = np.asarray(t32, dtype=np.float32)
    a = np.abs(t.astype(np.float64))
    out = np.empty(a.shape, dtype=np.uint8)
    for lo in range(0, a.size, 1 << 16):
        chunk = a.reshape(-1)[lo:lo + (1 << 16)]
        d = np.abs(chunk[:, None] - E4M3_POS[None, :])
        best = d.min(axis=1, keepdims=True)
        cand = d == best
        # among equally near codes prefer the even one (LSB of mantissa 0)
        even = cand & ((np.arange(0x7F) & 1) == 0)[None, :]
        pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        pick = np.where(chunk > 448.0, 0x7E, pick)
        out.reshape(-1)[lo:lo + (1 << 16)] = pick
    sign = (t.view(np.uint32) >> 31).astype(np.uint8)
    return out | (sign << 7)


def _parse_value(s):
    s = s.strip()
    if "0x" in s:
        return np.float32(float.fromhex(s))
    return np.float32(float(s))


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            vals, sb, codes, _why = [p.strip() for p in line.split(";", 3)]
            rows.append(([_parse_value(v) for v in vals.split(",")], int(sb, 16),
                         [int(c, 16) for c in codes.split(",")]))
    return rows


@pytest.mark.parametrize("vals,sb,codes", _golden_rows())
def test_golden_blocks(vals, sb, codes):
    y = np.zeros((1, 32), dtype=np.float32)
    y[0, :len(vals)] = vals
    q, s = O.mx_quantize_logical(y)
    assert s[0, 0] == sb
    assert list(q[0, :len(codes)]) == codes
    assert np.all(q[0, len(codes):] == 0)


def test_e4m3_encode_matches_brute_force():
    rng = np.random.default_rng(1)
    pts = []
    # dense sweep: every fp32 in [2^-12, 512) whose low 10 mantissa bits are zero
    base = np.arange(np.float32(2.0 ** -12).view(np.uint32), np.float32(512.0).view(np.uint32), 1024,
                     dtype=np.uint32)
    pts.append(base.view(np.float32))
    # every midpoint between neighbouring E4M3 values, and its fp32 neighbours
    mids = ((E4M3_POS[1:] + E4M3_POS[:-1]) / 2).astype(np.float32)
    pts += [mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))]
    pts += [E4M3_POS.astype(np.float32), np.float32([448, 449, 463.99997, 464, 464.00003, 479, 480, 511.99997])]
    # tiny and subnormal fp32 inputs, and random finite bit patterns
    pts.append(np.float32([0.0, 2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11, 2.0 ** -126, 2.0 ** -149, 1e-30]))
    rnd = rng.integers(0, 0x7F800000, size=200_000, dtype=np.uint32).view(np.float32)
    pts.append(rnd[np.abs(rnd) < 600])
    t = np.concatenate(pts).astype(np.float32)
    t = np.concatenate([t, -t])
    assert np.array_equal(O.e4m3_encode(t), _brute_e4m3(t))


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_e4m3_round_trip():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert len(codes) == 254
    back = O.e4m3_encode(O.e4m3_decode(codes).astype(np.float32))
    assert np.array_equal(back, codes)


def test_ue8m0_decode():
    b = np.arange(255, dtype=np.uint8)
    got = O.ue8m0_decode(b)
    for i in range(255):
        assert got[i] == math.ldexp(1.0, i - 127)
    assert np.isnan(O.ue8m0_decode(np.uint8([255]))[0])
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.from_numpy(b.copy()).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        assert np.array_equal(ref, got)


def test_power_of_two_amax():
    for k in range(-119, 128):
        y = np.zeros((1, 32), dtype=np.float32)
        y[0, 5] = np.float32(math.ldexp(1.0, k))
        q, s = O.mx_quantize_logical(y)
        assert s[0, 0] == k + 119
        assert q[0, 5] == 0x78                      # 2^k / 2^(k-8) = 256 = 1.0 * 2^8


def test_quantisation_error_bound():
    rng = np.random.default_rng(7)
    y = (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-30, 30, (64, 1)))).astype(np.float32)
    q, sb = O.mx_quantize_logical(y)
    e = sb.astype(np.int64) - 127
    t = y.reshape(64, 8, 32).astype(np.float64) / np.exp2(e)[:, :, None]
    deq = O.e4m3_decode(q).reshape(64, 8, 32)
    a = np.abs(t)
    # half the grid spacing at |t| (spacing 2^(floor(log2|t|)-3), >= 2^-9), or saturation
    ex = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    bound = np.where(a > 448.0, a - 448.0, np.exp2(ex - 4))
    assert np.all(np.abs(deq - t) <= bound + 0.0)
    # the scale puts every block's amax in [256, 512) after scaling
    amax = np.abs(t).max(axis=2)
    assert np.all((amax >= 256) & (amax < 512))


# ---------------------------------------------------------------------------
# norm
# ---------------------------------------------------------------------------

def _bf16_bits(a):
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_pairwise_tree_order():
    # leaves 1, 2^-24, 2^-24 at positions 0, 4096, 4097 of a 6144-wide row:
    # the tree adds the two small leaves first (exact 2^-23), then 1 + 2^-23;
    # a left-to-right sum would lose both (1 + 2^-24 rounds to 1, twice).
    v = np.zeros((1, 6144), dtype=np.float32)
    v[0, 0] = 1.0
    v[0, 4096] = v[0, 4097] = 2.0 ** -24
    assert O.pairwise_sum_f32(v)[0] == np.float32(1.0 + 2.0 ** -23)
    # leaves [1, 0, 2^-24, 2^-24]: (1+0) + (2^-24+2^-24) = 1 + 2^-23
    v = np.float32([[1.0, 0.0, 2.0 ** -24, 2.0 ** -24]])
    assert O.pairwise_sum_f32(v)[0] == np.float32(1.0 + 2.0 ** -23)


def test_pairwise_sum_error_bound():
    rng = np.random.default_rng(3)
    v = (rng.standard_normal((16, 6144)) ** 2).astype(np.float32)
    got = O.pairwise_sum_f32(v).astype(np.float64)
    exact = np.array([math.fsum(r) for r in v.astype(np.float64)])
    u = 2.0 ** -24
    assert np.all(np.abs(got - exact) <= math.ceil(math.log2(6144)) * u * exact)


def test_norm_closed_form_ones():
    # x = 1 everywhere, w = 0, eps = 1e-6: sum of squares 6144 exactly, r just
    # below 1, so every y = r in [0.5, 1): E = -1 - 8 = -9 (byte 118) and
    # t = r * 512 > 448 saturates every code to 0x7E.
    x = np.full((2, 6144), 0x3F80, dtype=np.uint16)         # bf16 1.0
    w = np.zeros(6144, dtype=np.uint16)
    assert O.pairwise_sum_f32(O.bf16_bits_to_f32(x) ** 2)[0] == 6144.0
    y = O.gemma_rmsnorm_f32(x, w, 1e-6)
    assert np.all(y < 1.0) and np.all(y > 0.9999)
    q, s = O.rmsnorm_quant(x, w, 1e-6)
    assert np.all(q == 0x7E)
    assert np.all(O.unswizzle_scales(s, 2, 192) == 0x76)


def test_norm_small_closed_form():
    # H = 32, x = [3, 4, 0, ...], eps = 0: mean(x^2) = 25/32, so
    # y_i = x_i * sqrt(32)/5 * (1 + w_i); compared with fp32 to a few ulp.
    x = np.zeros(32, dtype=np.float32)
    x[0], x[1] = 3.0, 4.0
    w = np.zeros(32, dtype=np.float32)
    w[0], w[1] = 1.0, -0.5
    y = O.gemma_rmsnorm_f32(_bf16_bits(x)[None], _bf16_bits(w), 0.0)[0]
    k = math.sqrt(32.0) / 5.0
    assert abs(y[0] - 3 * k * 2.0) <= 4 * 2.0 ** -23 * 3 * k * 2.0
    assert abs(y[1] - 4 * k * 0.5) <= 4 * 2.0 ** -23 * 4 * k * 0.5
    assert np.all(y[2:] == 0.0)


def test_norm_scale_invariance_eps0():
    # with eps = 0, scaling a row by 2^k leaves y, hence codes and scales, unchanged
    rng = np.random.default_rng(5)
    x = rng.standard_normal((8, 6144)).astype(np.float32)
    w = rng.uniform(-0.1, 0.1, 6144).astype(np.float32)
    q0, s0 = O.rmsnorm_quant(_bf16_bits(x), _bf16_bits(w), 0.0)
    for k in (-20, -3, 5, 30):
        q1, s1 = O.rmsnorm_quant(_bf16_bits(x * np.float32(2.0 ** k)), _bf16_bits(w), 0.0)
        assert np.array_equal(q0, q1) and np.array_equal(s0, s1)


def test_norm_against_float64_definition():
    rng = np.random.default_rng(11)
    xb = _bf16_bits(rng.standard_normal((32, 6144)).astype(np.float32) * 3)
    wb = _bf16_bits(rng.uniform(-0.1, 0.1, 6144).astype(np.float32))
    eps = 1e-2                                              # large enough to matter
    y = O.gemma_rmsnorm_f32(xb, wb, eps).astype(np.float64)
    x64 = O.bf16_bits_to_f32(xb).astype(np.float64)
    w64 = O.bf16_bits_to_f32(wb).astype(np.float64)
    eps32 = float(np.float32(eps))
    ref = x64 / np.sqrt(np.array([math.fsum(r) for r in x64 ** 2]) / 6144 + eps32)[:, None] * (1 + w64)
    assert np.max(np.abs(y - ref) / (np.abs(ref) + 1e-30)) < 8 * 2.0 ** -24


# ---------------------------------------------------------------------------
# BF16 form of the norm (sequence-parallel path)
# ---------------------------------------------------------------------------

def test_bf16_rounding_hand_values():
    # bf16 keeps 7 fraction bits: the spacing at 1.0 is 2^-7, so 1 + 2^-8 is a
    # tie (to even: 1.0) and 1 + 3*2^-8 is a tie (to even: 1 + 2^-6).
    v = np.array([1.0, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -20, -2.5, 3.0e38],
                 dtype=np.float32)
    got = O.f32_to_bf16_bits(v)
    assert got[0] == 0x3F80 and got[1] == 0x3F80 and got[2] == 0x3F82 and got[3] == 0x3F81
    assert got[4] == 0xC020                                # -2.5 is exact
    assert got[5] == 0x7F62                                # 0x7F61B1E6: low half above the tie


def test_bf16_rounding_matches_torch():
    # the library cast (round to nearest even) over random finite patterns,
    # a third of them exact ties
    rng = np.random.default_rng(17)
    u = rng.integers(0, 0xFF7FFFFF, size=200_000, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 0x7F7F, size=100_000, dtype=np.uint32) << 16) | 0x8000
    v = np.concatenate([u, ties, ties | 0x80000000]).view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) < 3.38e38)]            # no overflow to inf
    want = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f32_to_bf16_bits(v), want)


def test_bf16_rounding_is_nearest():
    # brute force: the result is the nearer of the two bf16 neighbours
    rng = np.random.default_rng(19)
    v = (rng.standard_normal(20_000) * 10.0 ** rng.integers(-30, 30, 20_000)).astype(np.float32)
    b = O.f32_to_bf16_bits(v)
    dec = O.bf16_bits_to_f32(b).astype(np.float64)
    lo = O.bf16_bits_to_f32((v.view(np.uint32) >> 16).astype(np.uint16)).astype(np.float64)
    hi = O.bf16_bits_to_f32(((v.view(np.uint32) >> 16) + 1).astype(np.uint16)).astype(np.float64)
    err = np.abs(dec - v.astype(np.float64))
    assert np.all(err <= np.minimum(np.abs(lo - v), np.abs(hi - v)))


def test_rmsnorm_bf16_closed_forms():
    # x = 2 everywhere, w = 0.5, eps = 0: mean(x^2) = 4, r = 1/2, y = 1.5 (0x3FC0)
    x = np.full((3, 512), 0x4000, dtype=np.uint16)          # bf16 2.0
    w = np.full(512, 0x3F00, dtype=np.uint16)               # bf16 0.5
    assert np.all(O.rmsnorm_bf16(x, w, 0.0) == 0x3FC0)
    # x = [3, 4, 0...] over H = 32, w = 0, eps = 0: y_0 = 3*sqrt(32)/5 = 3.394...
    x = np.zeros((1, 32), dtype=np.uint16)
    x[0, 0], x[0, 1] = 0x4040, 0x4080                       # 3.0, 4.0
    y = O.bf16_bits_to_f32(O.rmsnorm_bf16(x, np.zeros(32, dtype=np.uint16), 0.0))[0]
    assert abs(float(y[0]) - 3 * math.sqrt(32) / 5) <= 2.0 ** -7 * 2
    assert abs(float(y[1]) - 4 * math.sqrt(32) / 5) <= 2.0 ** -7 * 4
    assert np.all(y[2:] == 0.0)


def test_rmsnorm_bf16_within_half_ulp_of_norm():
    rng = np.random.default_rng(23)
    xb = _bf16_bits(rng.standard_normal((16, 6144)).astype(np.float32))
    wb = _bf16_bits(rng.uniform(-0.1, 0.1, 6144).astype(np.float32))
    y = O.gemma_rmsnorm_f32(xb, wb, 1e-6).astype(np.float64)
    yb = O.bf16_bits_to_f32(O.rmsnorm_bf16(xb, wb, 1e-6)).astype(np.float64)
    nz = y != 0
    ulp = 2.0 ** (np.floor(np.log2(np.abs(y[nz]))) - 7)
    assert np.all(np.abs(yb[nz] - y[nz]) <= ulp / 2)


# ---------------------------------------------------------------------------
# F8_128x4 layout
# ---------------------------------------------------------------------------

def test_swizzle_hand_values():
    c = 192                                                  # 6144 / 32
    assert O.swizzle_offset(0, 0, c) == 0
    assert O.swizzle_offset(0, 1, c) == 1
    assert O.swizzle_offset(0, 3, c) == 3
    assert O.swizzle_offset(1, 0, c) == 16
    assert O.swizzle_offset(31, 0, c) == 31 * 16
    assert O.swizzle_offset(32, 0, c) == 4
    assert O.swizzle_offset(96, 3, c) == 15
    assert O.swizzle_offset(0, 4, c) == 512
    assert O.swizzle_offset(128, 0, c) == 48 * 512
    assert O.swizzle_offset(129, 5, c) == 48 * 512 + 512 + 16 + 1
    assert O.scale_bytes(6144, 2048) == 6144 * 64
    assert O.scale_bytes(1, 32) == 128 * 4                   # one row, one block -> padded


def test_swizzle_is_block_transpose():
    # independent formulation: pad S to (Rp, Cp), view it as
    # [row block][row/32 within block][row % 32][column block][column % 4]
    # and store it as [row block][column block][row % 32][row/32][column % 4]
    rng = np.random.default_rng(2)
    for rows, c in [(128, 4), (300, 6), (1, 1), (257, 96), (1024, 64)]:
        s = rng.integers(1, 255, size=(rows, c), dtype=np.uint8)
        rp, cp = -(-rows // 128) * 128, -(-c // 4) * 4
        pad = np.zeros((rp, cp), dtype=np.uint8)
        pad[:rows, :c] = s
        ref = pad.reshape(rp // 128, 4, 32, cp // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)
        got = O.swizzle_scales(s)
        assert np.array_equal(got, ref)
        assert np.array_equal(O.unswizzle_scales(got, rows, c), s)
        assert got.size == O.scale_bytes(rows, c * 32)


# ---------------------------------------------------------------------------
# GEMM reference
# ---------------------------------------------------------------------------

def test_gemm_one_hot_selects_column():
    # B row n is the E4M3 value 1.0 (0x38) at column k_n with scale byte 127:
    # C[m, n] must be exactly A's decoded element (m, k_n) -- catches a
    # transposed operand or a misplaced scale.
    rng = np.random.default_rng(4)
    m, n, k = 130, 40, 96
    a_q = rng.integers(0, 256, size=(m, k), dtype=np.uint8)
    a_q[(a_q & 0x7F) == 0x7F] = 0x30
    a_sb = rng.integers(100, 150, size=(m, k // 32), dtype=np.uint8)
    kn = rng.integers(0, k, size=n)
    b_q = np.zeros((n, k), dtype=np.uint8)
    b_q[np.arange(n), kn] = 0x38
    b_sb = np.full((n, k // 32), 127, dtype=np.uint8)
    c = O.gemm_ref(a_q, O.swizzle_scales(a_sb), b_q, O.swizzle_scales(b_sb))
    expect = np.array([[O.e4m3_decode(a_q[i, kn[j]]) * 2.0 ** (int(a_sb[i, kn[j] // 32]) - 127)
                        for j in range(n)] for i in range(m)])
    assert np.array_equal(c, expect)


def test_gemm_decoded_vs_torch_casts():
    rng = np.random.default_rng(6)
    q = rng.integers(0, 256, size=(64, 128), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0
    sb = rng.integers(110, 140, size=(64, 4), dtype=np.uint8)
    got = O.mx_decode(q, O.swizzle_scales(sb))
    el = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64)
    sc = torch.from_numpy(sb).to(torch.float64).sub(127).exp2()
    ref = (el.view(64, 4, 32) * sc[:, :, None]).reshape(64, 128).numpy()
    assert np.array_equal(got, ref)


def test_gemm_vs_unquantised_brute_force():
    # tiny GEMM on the original bf16 values (triple loop over exact fractions)
    # against the oracle's decoded GEMM, within the elementwise quantisation bound
    rng = np.random.default_rng(8)
    m, n, k = 6, 5, 64
    a = O.bf16_bits_to_f32(_bf16_bits(rng.standard_normal((m, k)).astype(np.float32)))
    b = O.bf16_bits_to_f32(_bf16_bits((rng.standard_normal((n, k)) * 0.02).astype(np.float32)))
    aq, as_ = O.quant(_bf16_bits(a))
    bq, bs_ = O.quant(_bf16_bits(b))
    got = O.gemm_ref(aq, as_, bq, bs_)
    da = O.mx_decode(aq, as_)
    db = O.mx_decode(bq, bs_)

    def elem_bound(v, scale_blocks):
        # RNE error bound per element at the block's scale 2^E: half the E4M3 grid step
        e = scale_blocks.astype(np.int64) - 127
        t = np.abs(v).reshape(v.shape[0], -1, 32) / np.exp2(e)[:, :, None]
        ex = np.floor(np.log2(np.maximum(t, 2.0 ** -6)))
        half = np.where(t > 448, t - 448, np.exp2(ex - 4))
        return (half * np.exp2(e)[:, :, None]).reshape(v.shape)

    ea = elem_bound(a.astype(np.float64), O.unswizzle_scales(as_, m, 2))
    eb = elem_bound(b.astype(np.float64), O.unswizzle_scales(bs_, n, 2))
    assert np.all(np.abs(da - a) <= ea) and np.all(np.abs(db - b) <= eb)
    for i in range(m):
        for j in range(n):
            exact = sum(Fraction(float(a[i, kk])) * Fraction(float(b[j, kk])) for kk in range(k))
            bound = sum(abs(float(a[i, kk])) * eb[j, kk] + abs(float(b[j, kk])) * ea[i, kk]
                        + ea[i, kk] * eb[j, kk] for kk in range(k))
            assert abs(got[i, j] - float(exact)) <= bound * (1 + 1e-12) + 1e-300
    # and the quantisation actually changed something (the bound is not vacuous)
    assert np.max(np.abs(got - a.astype(np.float64) @ b.astype(np.float64).T)) > 0


def test_gemm_small_integer_exact():
    # small-integer E4M3 values with power-of-two scales: every product and
    # partial sum is exactly representable, so C equals the integer dot product
    rng = np.random.default_rng(9)
    m, n, k = 16, 24, 128
    ints = np.array([0, 1, 2, 3, 4, 5, 6, 7, 8, 10, 12, 16])
    ai = rng.choice(ints, size=(m, k)) * rng.choice([-1, 1], size=(m, k))
    bi = rng.choice(ints, size=(n, k)) * rng.choice([-1, 1], size=(n, k))
    aq = O.e4m3_encode(ai.astype(np.float32))
    bq = O.e4m3_encode(bi.astype(np.float32))
    one = np.full((m, k // 32), 127, np.uint8)
    two = np.full((n, k // 32), 128, np.uint8)                # every B block scaled by 2
    c = O.gemm_ref(aq, O.swizzle_scales(one), bq, O.swizzle_scales(two))
    assert np.array_equal(c, 2.0 * (ai @ bi.T))
