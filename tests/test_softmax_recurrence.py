"""The tile recurrence of the split-KV attention kernels, in float64 on the host.

The kernels walk a row's keys tile by tile, keeping a reference maximum m, a sum
l = sum 2^(s - m) and numerators O = sum 2^(s - m) v, and merge such states across warps
and CTAs by rescaling each to a common reference.  The cluster and q8_0 instances move m
only when a tile's maximum exceeds it by more than 2^8 (log2 units), so the probabilities
they round to F16 stay within [0, 256].  These tests check, with no rounding in the way,
that this recurrence and the merge give exactly the softmax-weighted average of the
values (the quantity the oracle computes directly), for the reference moved at every
growth (threshold 0) and lazily, and that the probability bound holds.  Scores are in the
log2 domain, as in the kernels (the scale log2(e)/sqrt(d) is applied before).
"""

import numpy as np
import pytest

LAZY = 8.0


def tile_states(s, v, tile, threshold):
    """Walk scores s[n] (with -inf for masked keys) and values v[n, d] in tiles; return the
    state (m, l, O) and the largest probability formed on the way."""
    m, l = -np.inf, 0.0
    o = np.zeros(v.shape[1])
    pmax = 0.0
    for a in range(0, len(s), tile):
        st, vt = s[a:a + tile], v[a:a + tile]
        mx = st.max()
        if mx > m + threshold:                       # move the reference (all -inf: never)
            mnew = max(m, mx)
            alpha = 1.0 if mnew == -np.inf else 2.0 ** (m - mnew)
            l *= alpha
            o *= alpha
            m = mnew
        muse = 0.0 if m == -np.inf else m
        p = 2.0 ** (st - muse)
        pmax = max(pmax, float(p.max(initial=0.0)))
        l += p.sum()
        o += p @ vt
    return m, l, o, pmax


def merge(states):
    """Log-sum-exp merge of (m, l, O) states to the largest reference, as the kernels'
    pre-merge, owner merge and combine kernel do."""
    mm = max(st[0] for st in states)
    muse = 0.0 if mm == -np.inf else mm
    l = sum(2.0 ** (st[0] - muse) * st[1] for st in states)
    o = sum(2.0 ** (st[0] - muse) * st[2] for st in states)
    return mm, l, o


def softmax_average(s, v):
    keep = np.isfinite(s)
    if not keep.any():
        return np.zeros(v.shape[1])
    w = 2.0 ** (s[keep] - s[keep].max())
    return (w / w.sum()) @ v[keep]


def scores(kind, n, rng):
    x = np.arange(n, dtype=np.float64)
    if kind == "random":
        s = rng.normal(0.0, 3.0, n)
    elif kind == "rising":                           # a new maximum in every tile
        s = 0.2 * x
    elif kind == "falling":                          # the maximum in the first key
        s = -0.2 * x
    elif kind == "staircase":                        # +7.46 per 64 keys: moves every other tile
        s = 7.46 * np.floor(x / 64)
    elif kind == "huge":                             # beyond float64's own exp range
        s = 3000.0 * np.sin(x / 50.0)
    elif kind == "sparse":                           # whole tiles masked
        s = rng.normal(0.0, 10.0, n)
        s[(x // 64) % 3 == 1] = -np.inf
        s[rng.random(n) < 0.2] = -np.inf
    else:
        raise ValueError(kind)
    return s


@pytest.mark.parametrize("kind", ["random", "rising", "falling", "staircase", "huge", "sparse"])
@pytest.mark.parametrize("threshold", [0.0, LAZY])
def test_tile_recurrence_and_merge_give_the_softmax(kind, threshold):
    rng = np.random.default_rng(7)
    n, d, tile = 64 * 37 + 19, 16, 64              # a ragged last tile
    s = scores(kind, n, rng)
    v = rng.normal(0.0, 1.0, (n, d))
    want = softmax_average(s, v)
    # one pass over everything, and the same keys split into uneven chunks merged after
    m, l, o, pmax = tile_states(s, v, tile, threshold)
    assert pmax <= 2.0 ** threshold * (1 + 1e-12)
    got = o / l if l > 0 else np.zeros(d)
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-12)
    cuts = [0, 5 * 64, 6 * 64 + 7, 20 * 64, 21 * 64, n]
    parts = [tile_states(s[a:b], v[a:b], tile, threshold)[:3] for a, b in zip(cuts, cuts[1:])]
    mm, ll, oo = merge(parts)
    got = oo / ll if ll > 0 else np.zeros(d)
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-12)


def test_lazy_reference_moves_rarely_on_ordinary_scores():
    # the reason for the lazy reference: on ordinary scores it moves on the first tile and
    # then almost never, where the running maximum moves on most tiles
    rng = np.random.default_rng(11)
    s = rng.normal(0.0, 2.0, 64 * 64)
    moves = {0.0: 0, LAZY: 0}
    for threshold in moves:
        m = -np.inf
        for a in range(0, len(s), 64):
            mx = s[a:a + 64].max()
            if mx > m + threshold:
                moves[threshold] += 1
                m = max(m, mx)
    assert moves[LAZY] == 1
    assert moves[0.0] > moves[LAZY]


def test_all_masked_rows_give_zero():
    v = np.ones((130, 4))
    s = np.full(130, -np.inf)
    for threshold in (0.0, LAZY):
        m, l, o, pmax = tile_states(s, v, 64, threshold)
        assert m == -np.inf and l == 0.0 and not o.any() and pmax == 0.0
        assert merge([(m, l, o), (m, l, o)])[1] == 0.0
