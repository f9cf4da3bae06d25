"""The sum of squares of a norm row, in the orders the CUDA kernels take it,
is the oracle's pairwise tree bit for bit (CPU, float32 numpy).

The kernels hold a 6144-element row as 24 chunks of 256; lane l of a warp
holds elements [256c + 8l, +8) of chunk c.  Two orders are used:
  * per chunk: an in-lane tree of 8 squares, a 5-level xor butterfly across
    the lanes, then the chunk tree (chunks 0-15 and 16-23, then their sum);
  * reduce-scatter: the same in-lane trees; at the three lane levels below
    8 lanes each lane keeps half of its chunk partials and adds its partner's
    half of the same chunks; two more butterfly levels finish the chunks
    held by each lane (c = l mod 8), three more combine chunks 8k..8k+7.
Both must reach exactly the nodes of the oracle's pairwise tree (its reading
R2: the pages name the Gemma RMSNorm, vLLM PR #64659, Details, but no
summation order), so that the codes the GPU writes can match the oracle byte
for byte.  These tests check that claim on the CPU, with inputs spread over a
wide exponent range so that any other association changes low-order bits.
"""

import numpy as np

import oracle as O

H, LANES, CHUNK = 6144, 32, 256
NCH = H // CHUNK


def _rows(seed, m=48):
    rng = np.random.default_rng(seed)
    mant = rng.uniform(1.0, 2.0, size=(m, H))
    expo = rng.integers(-20, 21, size=(m, H))
    sign = rng.choice([-1.0, 1.0], size=(m, H))
    return (sign * mant * np.exp2(expo)).astype(np.float32)


def _lane_trees(x):
    """(rows, NCH, LANES) float32: each lane's 8 squares, ((e0+e1)+(e2+e3))+((e4+e5)+(e6+e7))."""
    sq = (x * x).astype(np.float32).reshape(x.shape[0], NCH, LANES, 8)
    l1 = sq[..., 0::2] + sq[..., 1::2]
    l2 = l1[..., 0::2] + l1[..., 1::2]
    return l2[..., 0] + l2[..., 1]


def _xor_partner(a, m):
    """Value of lane l ^ m, for every lane (last axis)."""
    return a[..., np.arange(LANES) ^ m]


def _per_chunk_order(x):
    p = _lane_trees(x)
    for m in (1, 2, 4, 8, 16):
        p = p + _xor_partner(p, m)
    lvl = p[..., 0].reshape(-1, NCH // 8, 8)            # chunk sums (identical in every lane), 3 groups of 8
    while lvl.shape[2] > 1:                             # the tree inside each 8-chunk group
        lvl = lvl[..., 0::2] + lvl[..., 1::2]
    t = lvl[..., 0]                                     # (rows, 3): chunks 0-7, 8-15, 16-23
    return (t[:, 0] + t[:, 1]) + t[:, 2]


def _reduce_scatter_order(x):
    v = _lane_trees(x)                                  # (rows, NCH, LANES)
    lane = np.arange(LANES)
    for level, m in enumerate((1, 2, 4)):
        b = ((lane >> level) & 1).astype(bool)          # which half of its partials a lane keeps
        even, odd = v[:, 0::2, :], v[:, 1::2, :]
        keep = np.where(b, odd, even)
        give = np.where(b, even, odd)
        v = keep + _xor_partner(give, m)
    # lane l now holds, for k = 0..2, the 64-element sum of chunk 8k + (l & 7)
    for m in (8, 16, 1, 2, 4):
        v = v + _xor_partner(v, m)
    u = v[..., 0]                                       # chunks 8k..8k+7, identical in every lane
    return (u[:, 0] + u[:, 1]) + u[:, 2]


def _oracle(x):
    return O.pairwise_sum_f32((x * x).astype(np.float32))


def test_reduce_scatter_holds_chunk_8k_plus_lane():
    # after the three reduce-scatter levels lane l holds the 64-element sums of
    # chunks 8k + (l & 7): check against sums taken directly
    x = _rows(1, m=4)
    v = _lane_trees(x)
    lane = np.arange(LANES)
    for level, m in enumerate((1, 2, 4)):
        b = ((lane >> level) & 1).astype(bool)
        keep = np.where(b, v[:, 1::2, :], v[:, 0::2, :])
        give = np.where(b, v[:, 0::2, :], v[:, 1::2, :])
        v = keep + _xor_partner(give, m)
    full = _lane_trees(x)
    for l in range(LANES):
        g = l & ~7
        for k in range(NCH // 8):
            c = 8 * k + (l & 7)
            sub = full[:, c, g:g + 8]                   # the 8 lanes of l's group, in lane order
            ref = (((sub[:, 0] + sub[:, 1]) + (sub[:, 2] + sub[:, 3]))
                   + ((sub[:, 4] + sub[:, 5]) + (sub[:, 6] + sub[:, 7])))
            assert np.array_equal(v[:, k, l], ref)


def test_per_chunk_order_is_the_pairwise_tree():
    for seed in range(4):
        x = _rows(seed)
        assert np.array_equal(_per_chunk_order(x), _oracle(x))


def test_reduce_scatter_order_is_the_pairwise_tree():
    for seed in range(4):
        x = _rows(100 + seed)
        assert np.array_equal(_reduce_scatter_order(x), _oracle(x))


def test_inputs_separate_orders():
    # the inputs are wide enough that a different association is visible:
    # a left-to-right sum differs from the tree on most rows
    x = _rows(7)
    sq = (x * x).astype(np.float32)
    seq = np.zeros(x.shape[0], dtype=np.float32)
    for i in range(H):
        seq = seq + sq[:, i]
    assert np.mean(seq != _oracle(x)) > 0.5
