"""The sum of squares of a norm row in the order the lane-block kernels take
it, for every width they take and every (warps per row, chunks per warp)
shape the kernel choice can give them, is the oracle's pairwise tree bit for
bit (CPU, float32 numpy).

The lane-block kernels cut a row into 1024-element chunks (the last one
zero-padded): lane l holds the 32-element block [32 l, +32) of each chunk.
  * a lane's 32 squares form a subtree of the pairwise tree, and a 5-level
    xor butterfly across the lanes completes the chunk: each chunk total is
    the pairwise tree of its 1024 (padded) squares;
  * a warp holds a run of NCW chunks (chunks past the row are zeros) and
    combines their totals with a binary counter: the total of chunk c is
    added to the pending subtree of each lower level whose bit of c is set,
    and the pending subtrees of NCW's set bits are finally added from the
    lowest level up;
  * WPR warps hold consecutive runs, combined in the order the kernel writes
    for each warp count: (t0+t1), (t0+t1)+t2, (t0+t1)+(t2+t3),
    ((t0+t1)+(t2+t3))+(t4+t5), and the full tree of eight.
The oracle pads the row with +0.0 to a power of two and adds sibling pairs
level by level (its reading of the unstated summation order).  Inputs span
2^-20..2^20, so any other association changes low-order bits."""

import numpy as np
import pytest

import mxfp8_norm_quant_gb300 as mx
import oracle as O

SMS = 152


def _rows(h, seed, m=6):
    rng = np.random.default_rng(seed)
    mant = rng.uniform(1.0, 2.0, size=(m, h))
    expo = rng.integers(-20, 21, size=(m, h))
    sign = rng.choice([-1.0, 1.0], size=(m, h))
    return (sign * mant * np.exp2(expo)).astype(np.float32)


def _pairwise(v):
    """Pairwise tree over the last axis (a power of two long), float32."""
    while v.shape[-1] > 1:
        v = (v[..., 0::2] + v[..., 1::2]).astype(np.float32)
    return v[..., 0]


def _lane_block_order(x, wpr, ncw):
    m, h = x.shape
    nch = wpr * ncw
    sq = np.zeros((m, nch * 1024), dtype=np.float32)
    sq[:, :h] = (x * x).astype(np.float32)
    lane = _pairwise(sq.reshape(m, nch, 32, 32))             # (m, nch, lanes): each lane's block
    for b in (1, 2, 4, 8, 16):                               # the butterfly across the lanes
        lane = (lane + lane[..., np.arange(32) ^ b]).astype(np.float32)
    chunk = lane[..., 0]                                     # (m, nch): identical in every lane
    warp = []
    for w in range(wpr):
        lvl = {}
        for c in range(ncw):
            t = chunk[:, w * ncw + c]
            k = 0
            while (c >> k) & 1:
                t = (lvl[k] + t).astype(np.float32)
                k += 1
            lvl[k] = t
        ss = None
        for k in range(4):
            if (ncw >> k) & 1:
                ss = lvl[k] if ss is None else (lvl[k] + ss).astype(np.float32)
        warp.append(ss)
    t = warp
    f = lambda a, b: (a + b).astype(np.float32)
    if wpr == 1:
        return t[0]
    if wpr == 2:
        return f(t[0], t[1])
    if wpr == 3:
        return f(f(t[0], t[1]), t[2])
    if wpr == 4:
        return f(f(t[0], t[1]), f(t[2], t[3]))
    if wpr == 6:
        return f(f(f(t[0], t[1]), f(t[2], t[3])), f(t[4], t[5]))
    assert wpr == 8
    return f(f(f(t[0], t[1]), f(t[2], t[3])), f(f(t[4], t[5]), f(t[6], t[7])))


def _shapes():
    """Every (H, wpr, ncw) the kernel choice gives a lane-block kernel."""
    counts = sorted({1, 2, 100, 1000, 10**5} | {int(t * SMS) + d for t in (1, 1.5, 1.7, 2, 4, 4.65, 8, 16, 40.4, 64)
                                                 for d in (0, 1)})
    out = set()
    for h in range(64, 16385, 64):
        for m in counts:
            for form in (mx.MX_NORM_SWIZZLED, mx.MX_NORM_ROW_MAJOR, mx.MX_NORM_BF16):
                wpr, ncw, _, _ = mx.mx_rmsnorm_plan(m, h, form, SMS)
                if wpr:
                    out.add((h, wpr, ncw))
    return sorted(out)


def test_every_lane_block_shape_is_the_pairwise_tree():
    shapes = _shapes()
    assert len({(w, n) for _, w, n in shapes}) >= 10        # the table's variety is all there
    for h, wpr, ncw in shapes:
        x = _rows(h, seed=h * 16 + wpr * 4 + ncw)
        want = O.pairwise_sum_f32((x * x).astype(np.float32))
        got = _lane_block_order(x, wpr, ncw)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (h, wpr, ncw)


@pytest.mark.parametrize("h", [4096, 6144, 12288])
def test_inputs_separate_orders(h):
    # a left-to-right sum of the chunk totals (instead of the tree) differs
    # on these inputs, so the test above would catch a wrong combine order
    x = _rows(h, seed=7, m=32)
    want = O.pairwise_sum_f32((x * x).astype(np.float32))
    sq = np.zeros((x.shape[0], -(-h // 1024) * 1024), dtype=np.float32)
    sq[:, :h] = x * x
    chunks = _pairwise(sq.reshape(x.shape[0], -1, 1024))
    seq = chunks[:, 0]
    for c in range(1, chunks.shape[1]):
        seq = (seq + chunks[:, c]).astype(np.float32)
    assert not np.array_equal(seq.view(np.uint32), want.view(np.uint32))
