"""Pins of the float64 oracle against what the pages and mathematics fix.

Every check here compares the oracle with something other than itself: values printed
on the pages, hand-computed tiny cases, IEEE/RoPE closed forms, invariants and brute
force.  No GPU involved.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import ring_oracle as orc
from tests.conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# geometry: the printed Luce log values
# ---------------------------------------------------------------------------

def test_geometry_matches_printed_values():
    for c in _golden("geometry.json")["cases"]:
        g = orc.geometry(c["cap"], c["q_len"], c["head_dim"], c["n_head_kv"], c["n_layer"])
        assert g["kv_total"] == c["kv_total"]
        assert g["a_step"] == c["a_step"]
        assert g["kv_row"] == c["kv_row"]
        assert f"{g['cache_bytes'] / 2**20:.1f}" == c["cache_mib_1dp"]


def test_geometry_hand_values_other_caps():
    # cap 64, q 8: trash 64 + 8 = 72; kv_total = align_up(73, 32) = 96
    g = orc.geometry(64, 8, 128, 8, 1)
    assert (g["a_step"], g["trash_slot"], g["kv_total"]) == (18, 72, 96)
    # cap 32768, q 8: align_up(32777, 32) = 32800
    g = orc.geometry(32768, 8, 128, 8, 5)
    assert (g["trash_slot"], g["kv_total"]) == (32776, 32800)
    # 84,541,440 bytes = 2 * 5 * 1024 * 4128 * 2
    assert orc.geometry(4096, 8, 128, 8, 5)["cache_bytes"] == 84_541_440


# ---------------------------------------------------------------------------
# slot map, window arithmetic and masks: hand-computed tiny rings
# ---------------------------------------------------------------------------

def _tiny_ring(cap, q_len, swa):
    # head_dim 2, one kv head, one query head, one layer: only the bookkeeping matters
    return orc.RingOracle(cap, q_len, 2, 1, 1, 1, 10000.0, swa_window=swa)


def _rows(first, last, width=2):
    """Zero K rows; V rows carry their position exactly as (p mod 1024, p div 1024)."""
    n = last - first
    p = np.arange(first, last)
    k = np.zeros((1, n, width), np.float16)
    v = np.zeros((1, n, width), np.float16)
    v[0, :, 0] = p % 1024
    v[0, :, 1] = p // 1024
    return k, v


@pytest.mark.parametrize("case", _golden("tiny_ring.json")["cases"], ids=lambda c: c["name"])
def test_tiny_ring_hand_cases(case):
    cap, q_len, swa = case["cap"], case["q_len"], case["swa_window"]
    r = _tiny_ring(cap, q_len, swa)
    geo = case["geometry"]
    assert (r.a_step, r.trash_slot, r.kv_total) == (geo["a_step"], geo["trash_slot"],
                                                    geo["kv_total"])
    for st in case["steps"]:
        c = st["committed"]
        win, lo, start, n_new = orc.step_window(c, r.next_pos, cap)
        assert (win, lo, start, n_new) == (st["win"], st["lo"], st["start"], st["n_new"])
        k, v = _rows(start, c)
        path = r.begin_step(c, k, v, start)
        assert path == st["path"]
        assert r.slot_pos.tolist() == st["slot_pos"]
        mf = r.mask_full()
        for i in range(q_len):
            assert np.flatnonzero(mf[i] == 0).tolist() == st["visible_full"]
        assert set(np.unique(mf)) <= {0.0, -np.inf}
        if swa:
            assert orc.swa_low(c, cap, swa) == st["swa_lo"]
            ms = r.mask_swa()
            for i in range(q_len):
                assert np.flatnonzero(ms[i] == 0).tolist() == st["visible_swa"][i]


def test_slot_pos_brute_force_and_window_invariant():
    """slot_pos[s] = largest position ever stored with p % cap == s (else -1), and the
    visible slots hold exactly the positions [lo, c), each once."""
    rng = np.random.default_rng(7)
    for cap in (5, 16, 64):
        r = _tiny_ring(cap, 3, 0)
        stored = set()
        c = 0
        for _ in range(120):
            c += int(rng.choice([0, 1, 2, 5, 9, cap - 1, cap + 3, 3 * cap]))
            _, lo, start, _ = orc.step_window(c, r.next_pos, cap)
            k, v = _rows(start, c)
            r.begin_step(c, k, v, start)
            stored.update(range(start, c))
            for s in range(cap):
                cands = [p for p in stored if p % cap == s]
                assert r.slot_pos[s] == (max(cands) if cands else -1)
            mf = r.mask_full()
            vis = sorted(int(r.slot_pos[s]) for s in range(cap) if mf[0, s] == 0)
            assert vis == list(range(lo, c))
            # V rows carry their position: the visible slots hold exactly those rows
            for s in range(cap):
                if mf[0, s] == 0:
                    held = int(r.v[0, s, 0]) + 1024 * int(r.v[0, s, 1])
                    assert held == r.slot_pos[s]


def test_mask_counts_closed_form():
    rng = np.random.default_rng(3)
    cap, q = 32, 4
    for swa in (1, 7, 32, 50):
        r = _tiny_ring(cap, q, swa)
        c = 0
        for _ in range(60):
            c += int(rng.integers(0, 40))
            _, _, start, _ = orc.step_window(c, r.next_pos, cap)
            k, v = _rows(start, c)
            r.begin_step(c, k, v, start)
            win = min(c, cap)
            mf, ms = r.mask_full(), r.mask_swa()
            for i in range(q):
                assert int((mf[i, :cap] == 0).sum()) == win
                assert int((mf[i, cap:cap + q] == 0).sum()) == q
                assert int((ms[i, :cap] == 0).sum()) == min(swa, win)
                assert int((ms[i, cap:cap + q] == 0).sum()) == i + 1
                assert np.all(mf[i, cap + q:] == -np.inf) and np.all(ms[i, cap + q:] == -np.inf)


def test_empty_context_only_noise_visible():
    r = _tiny_ring(8, 2, 3)
    r.begin_step(0, np.zeros((1, 0, 2), np.float16), np.zeros((1, 0, 2), np.float16), 0)
    assert r.last_path == "fold"
    assert np.flatnonzero(r.mask_full()[0] == 0).tolist() == [8, 9]
    assert np.flatnonzero(r.mask_swa()[0] == 0).tolist() == [8]
    assert np.flatnonzero(r.mask_swa()[1] == 0).tolist() == [8, 9]


def test_pad_rows_leave_trash_zero_and_untouched_slots():
    r = _tiny_ring(8, 2, 0)
    r.k[:] = 1.0                                   # sentinel in every slot
    r.v[:] = 1.0
    k, v = _rows(0, 3)
    r.begin_step(3, k, v, 0)                       # fold: 3 real rows, 3 pads
    assert np.all(r.k[0, r.trash_slot] == 0) and np.all(r.v[0, r.trash_slot] == 0)
    assert np.all(r.v[0, 3:8] == 1.0)              # slots not written keep their value


def test_backwards_commit_and_short_rows_rejected():
    r = _tiny_ring(8, 2, 0)
    k, v = _rows(0, 5)
    r.begin_step(5, k, v, 0)
    with pytest.raises(ValueError):
        r.begin_step(4, k, v, 0)
    k, v = _rows(7, 9)
    with pytest.raises(ValueError):                # rows start at 7 but start is 5
        r.begin_step(9, k, v, 7)


# ---------------------------------------------------------------------------
# F16 storage rounding
# ---------------------------------------------------------------------------

def test_f16_round_to_nearest_even():
    for c in _golden("f16_rne.json")["cases"]:
        with np.errstate(over="ignore"):
            got = orc.to_f16(np.float64(c["x"])).view(np.uint16)
        assert int(got) == int(c["bits"], 16), c


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def test_rope_golden_values():
    for c in _golden("rope_neox.json")["cases"]:
        got = orc.rope_neox(np.array(c["x"], np.float64), c["pos"], c["theta"])
        np.testing.assert_allclose(got, c["expect"], rtol=0, atol=1e-15)


def test_rope_invariants():
    rng = np.random.default_rng(11)
    d = 128
    q = rng.standard_normal(d)
    k = rng.standard_normal(d)
    # identity at 0, pair norms preserved
    np.testing.assert_array_equal(orc.rope_neox(q, 0, 1e6), q)
    r = orc.rope_neox(q, 123457, 1e6)
    np.testing.assert_allclose(r[:64] ** 2 + r[64:] ** 2, q[:64] ** 2 + q[64:] ** 2, rtol=1e-12)
    # the score depends only on the position difference
    for m, n, t in [(5, 3, 100), (131000, 130000, 7), (0, 9, 4096)]:
        a = orc.rope_neox(q, m, 1e6) @ orc.rope_neox(k, n, 1e6)
        b = orc.rope_neox(q, m + t, 1e6) @ orc.rope_neox(k, n + t, 1e6)
        assert abs(a - b) < 1e-9 * (1 + abs(a))


def test_rope_rows_same_angle_for_every_head():
    rng = np.random.default_rng(2)
    rows = rng.standard_normal((3, 4 * 8))
    pos = np.array([0, 5, 77])
    out = orc.rope_rows(rows, pos, 4, 8, 10000.0)
    for h in range(4):
        np.testing.assert_array_equal(out[:, h * 8:(h + 1) * 8],
                                      orc.rope_neox(rows[:, h * 8:(h + 1) * 8], pos, 10000.0))


# ---------------------------------------------------------------------------
# attention: closed forms
# ---------------------------------------------------------------------------

def _positional_ring(cap, q_len, swa, d=4, n_head_kv=2, n_head=4):
    return orc.RingOracle(cap, q_len, d, n_head_kv, n_head, 1, 10000.0, swa_window=swa)


def _pos_rows(first, last, kv_row):
    n = last - first
    k = np.zeros((1, n, kv_row), np.float16)
    v = np.repeat(np.arange(first, last, dtype=np.float16)[None, :, None], kv_row, axis=2)
    return k, v


@pytest.mark.parametrize("kind", ["full", "swa"])
def test_zero_query_gives_mean_of_visible_positions(kind):
    """Q = 0 makes every visible key equally likely; with V rows holding their own
    position the output is the mean position of the visible set."""
    cap, q_len, swa = 16, 4, 6
    r = _positional_ring(cap, q_len, swa)
    c = 0
    for inc in [3, 9, 1, 20, 4, 33, 2]:
        c += inc
        _, lo, start, _ = orc.step_window(c, r.next_pos, cap)
        k, v = _pos_rows(start, c, r.kv_row)
        r.begin_step(c, k, v, start)
        kn = np.zeros((q_len, r.kv_row), np.float16)
        vn = np.repeat(np.arange(c, c + q_len, dtype=np.float16)[:, None], r.kv_row, axis=1)
        q = np.zeros((q_len, r.n_head, r.head_dim))
        o = r.attend(0, q, kn, vn, kind)
        for i in range(q_len):
            if kind == "full":
                want = (lo + c + q_len - 1) / 2.0          # {lo..c-1} U {c..c+q-1}
            else:
                slo = c - min(swa, min(c, cap))
                want = (slo + c + i) / 2.0                 # {slo..c-1} U {c..c+i}
            np.testing.assert_allclose(o[i], want, rtol=0, atol=1e-12)


def test_single_visible_key_returns_its_value():
    r = _positional_ring(8, 3, 2)
    r.begin_step(0, np.zeros((1, 0, r.kv_row), np.float16),
                 np.zeros((1, 0, r.kv_row), np.float16), 0)
    rng = np.random.default_rng(5)
    q = rng.standard_normal((3, r.n_head, r.head_dim)) * 3
    kn = rng.standard_normal((3, r.kv_row)).astype(np.float16)
    vn = rng.standard_normal((3, r.kv_row)).astype(np.float16)
    o = r.attend(0, q, kn, vn, "swa")
    for h in range(r.n_head):
        g = h // 2
        np.testing.assert_array_equal(o[0, h], vn[0, g * 4:(g + 1) * 4].astype(np.float64))


def test_softmax_scale_is_one_over_sqrt_head_dim():
    """Two visible noise keys; their score gap is ln 3 only if scale = 1/sqrt(d).

    Query row 0 and noise key 0 both sit at position 0 (committed = 0), where RoPE is
    the identity, so the stored F16 key is exactly (1, 0, ...)."""
    d = 16
    r = orc.RingOracle(8, 2, d, 1, 1, 1, 10000.0)
    r.begin_step(0, np.zeros((1, 0, d), np.float16), np.zeros((1, 0, d), np.float16), 0)
    a = 4.0 * math.log(3.0)                       # a * 1 / sqrt(16) = ln 3
    q = np.zeros((2, 1, d))
    q[0, 0, 0] = a
    kn = np.zeros((2, d), np.float16)
    kn[0, 0] = 1.0
    vn = np.zeros((2, d), np.float16)
    vn[0, :] = 5.0
    vn[1, :] = 1.0
    o = r.attend(0, q, kn, vn, "full")
    np.testing.assert_allclose(o[0, 0], 0.75 * 5.0 + 0.25 * 1.0, rtol=0, atol=1e-12)


def test_gqa_head_map():
    """Q = 0 and V = (kv head index + 1): query head h must read kv head h // G."""
    r = orc.RingOracle(8, 2, 4, 2, 8, 1, 10000.0)      # G = 4
    k = np.zeros((1, 5, 8), np.float16)
    v = np.zeros((1, 5, 8), np.float16)
    v[..., 0:4] = 1.0
    v[..., 4:8] = 2.0
    r.begin_step(5, k, v, 0)
    vn = np.zeros((2, 8), np.float16)
    vn[:, 0:4] = 1.0
    vn[:, 4:8] = 2.0
    o = r.attend(0, np.zeros((2, 8, 4)), np.zeros((2, 8), np.float16), vn, "full")
    for h in range(8):
        np.testing.assert_allclose(o[:, h], h // 4 + 1.0, atol=1e-12)


def test_masked_attention_core_closed_form():
    # weights exp(2)/(exp(2)+exp(0)) and the complement, with one masked key ignored
    q = np.array([[2.0, 0.0]])
    k = np.array([[1.0, 0.0], [0.0, 0.0], [50.0, 0.0]])
    v = np.array([[1.0, 0.0], [0.0, 1.0], [9.0, 9.0]])
    mask = np.array([[0.0, 0.0, -np.inf]])
    w = math.exp(2) / (math.exp(2) + 1)
    np.testing.assert_allclose(orc.masked_attention(q, k, v, mask, 1.0), [[w, 1 - w]],
                               atol=1e-15)


@pytest.mark.parametrize("kind", ["full", "swa"])
def test_dense_route_zero_query_closed_form(kind):
    """The dense-window route on its own: with Q = 0 and V rows holding their position,
    every output is the mean position of exactly the window plus the visible noise."""
    cap, q_len, swa, d, hkv, nh = 16, 4, 6, 4, 2, 4

    def rows_fn(pos):
        pos = np.asarray(pos)
        k = np.zeros((len(pos), hkv * d), np.float16)
        v = np.repeat(pos.astype(np.float16)[:, None], hkv * d, axis=1)
        return k, v

    for c in (0, 3, 16, 40, 41):
        kn = np.zeros((q_len, hkv * d), np.float16)
        vn = np.repeat(np.arange(c, c + q_len, dtype=np.float16)[:, None], hkv * d, axis=1)
        o = orc.attend_dense(c, cap, rows_fn, np.zeros((q_len, nh, d)), kn, vn, d, hkv, nh,
                             10000.0, kind=kind, swa_window=swa)
        for i in range(q_len):
            if kind == "full":
                want = (c - min(c, cap) + c + q_len - 1) / 2.0
            else:
                want = (c - min(swa, min(c, cap)) + c + i) / 2.0
            np.testing.assert_allclose(o[i], want, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# context-row producer: k_norm(W_k x), W_v x (readings P1-P3)
# ---------------------------------------------------------------------------

def test_k_norm_special_cases():
    """eps = 0: a constant head maps to w; a head with one non-zero entry a at index j
    maps to sign(a) sqrt(head_dim) w_j there and 0 elsewhere; scaling a head changes
    nothing; heads are normalised one by one (each head's mean square becomes 1)."""
    d, nh = 8, 3
    w = np.array([1.0, 2.0, -1.0, 0.5, 3.0, 1.5, -2.0, 0.25])
    x = np.concatenate([np.full(d, 7.0), np.zeros(d), np.full(d, -0.5)])
    x[d + 5] = -3.0
    y = orc.rms_norm_heads(x, w, 0.0, nh, d)
    np.testing.assert_allclose(y[:d], w, rtol=0, atol=1e-15)
    e = np.zeros(d)
    e[5] = -math.sqrt(d) * w[5]
    np.testing.assert_allclose(y[d:2 * d], e, rtol=0, atol=1e-14)
    np.testing.assert_allclose(y[2 * d:], -w, rtol=0, atol=1e-15)
    rng = np.random.default_rng(5)
    z = rng.standard_normal((4, nh * d)) * np.array([1e-3] * d + [1.0] * d + [1e3] * d)
    one = np.ones(d)
    yz = orc.rms_norm_heads(z, one, 0.0, nh, d).reshape(4, nh, d)
    np.testing.assert_allclose(np.mean(yz * yz, axis=-1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(orc.rms_norm_heads(z * 37.5, one, 0.0, nh, d),
                               orc.rms_norm_heads(z, one, 0.0, nh, d), rtol=1e-13)


def test_k_norm_epsilon_inside_the_root():
    """A head whose mean square equals eps is divided by sqrt(2 eps)."""
    d = 4
    x = np.full(d, 1e-3)                       # mean square 1e-6
    y = orc.rms_norm_heads(x, np.ones(d), 1e-6, 1, d)
    np.testing.assert_allclose(y, 1e-3 / math.sqrt(2e-6), rtol=1e-14)


def test_producer_brute_force_small_integers():
    """Small integer features and weights: every product is exact, so V equals the
    brute-force triple loop exactly; K's heads each have mean square 1 (w = 1, eps = 0)
    and point the same way as the brute-force projection."""
    rng = np.random.default_rng(11)
    n, hidden, nh, d = 5, 12, 2, 4
    feat = rng.integers(-2, 3, (n, hidden)).astype(np.float16)
    wk = rng.integers(-1, 2, (nh * d, hidden)).astype(np.float16)
    wv = rng.integers(-1, 2, (nh * d, hidden)).astype(np.float16)
    k, v = orc.produce_rows(feat, wk, wv, np.ones(d), 0.0, nh, d)
    for r in range(n):
        for o in range(nh * d):
            acc_v = 0.0
            acc_k = 0.0
            for i in range(hidden):
                acc_v += float(feat[r, i]) * float(wv[o, i])
                acc_k += float(feat[r, i]) * float(wk[o, i])
            assert float(v[r, o]) == acc_v
    kb = np.array([[sum(float(feat[r, i]) * float(wk[o, i]) for i in range(hidden))
                    for o in range(nh * d)] for r in range(n)]).reshape(n, nh, d)
    kk = k.reshape(n, nh, d)
    for r in range(n):
        for h in range(nh):
            if np.any(kb[r, h]):
                np.testing.assert_allclose(np.mean(kk[r, h] ** 2), 1.0, rtol=1e-13)
                cosang = kk[r, h] @ kb[r, h] / (np.linalg.norm(kk[r, h]) * np.linalg.norm(kb[r, h]))
                np.testing.assert_allclose(cosang, 1.0, rtol=1e-13)


def test_producer_permutation_weights_pick_features():
    """W_v a permutation matrix (not symmetric): V row = the permuted features, exactly."""
    hidden = 8
    perm = np.array([3, 0, 6, 1, 7, 2, 5, 4])
    P = np.zeros((hidden, hidden), np.float16)
    P[np.arange(hidden), perm] = 1.0
    feat = (np.arange(2 * hidden, dtype=np.float64).reshape(2, hidden) - 5.0).astype(np.float16)
    _, v = orc.produce_rows(feat, P, P, np.ones(4), 0.0, 2, 4)
    np.testing.assert_array_equal(v, feat[:, perm])


def test_noise_projection_small_integers_and_heads():
    """F1: with small integers every product is exact: V noise equals the brute-force
    triple loop, K noise rounds the unit-RMS heads of W_k h to F16, and every query head
    of Q has mean square 1 (weights 1, eps 0) and points along the brute-force W_q h."""
    rng = np.random.default_rng(21)
    q_len, hidden, nh, nkv, d = 3, 10, 4, 2, 4
    h = rng.integers(-2, 3, (q_len, hidden)).astype(np.float16)
    wq = rng.integers(-1, 2, (nh * d, hidden)).astype(np.float16)
    wk = rng.integers(-1, 2, (nkv * d, hidden)).astype(np.float16)
    wv = rng.integers(-1, 2, (nkv * d, hidden)).astype(np.float16)
    q, k, v = orc.project_noise(h, wq, wk, wv, np.ones(d), np.ones(d), 0.0, nh, nkv, d)
    assert q.shape == (q_len, nh, d) and k.dtype == np.float16 and v.dtype == np.float16
    for r in range(q_len):
        for o in range(nkv * d):
            assert float(v[r, o]) == sum(float(h[r, i]) * float(wv[o, i]) for i in range(hidden))
        qb = np.array([sum(float(h[r, i]) * float(wq[o, i]) for i in range(hidden))
                       for o in range(nh * d)]).reshape(nh, d)
        for hh in range(nh):
            if np.any(qb[hh]):
                np.testing.assert_allclose(np.mean(q[r, hh] ** 2), 1.0, rtol=1e-13)
                cosang = q[r, hh] @ qb[hh] / (np.linalg.norm(q[r, hh]) * np.linalg.norm(qb[hh]))
                np.testing.assert_allclose(cosang, 1.0, rtol=1e-13)
        kb = np.array([sum(float(h[r, i]) * float(wk[o, i]) for i in range(hidden))
                       for o in range(nkv * d)]).reshape(nkv, d)
        for g in range(nkv):
            if np.any(kb[g]):
                kk = k[r].reshape(nkv, d)[g].astype(np.float64)
                np.testing.assert_allclose(np.mean(kk ** 2), 1.0, rtol=2e-3)    # F16 rounding


def test_noise_projection_query_weight_per_head():
    """F1: q_norm scales each query head's slice by its weight, element by element:
    with W_q a permutation and unit-RMS features the head values are w times the features."""
    d, nh, hidden = 4, 2, 8
    perm = np.array([5, 2, 7, 0, 1, 6, 3, 4])
    P = np.zeros((hidden, hidden), np.float16)
    P[np.arange(hidden), perm] = 1.0
    h = np.array([[1.0, -1.0, 1.0, -1.0, 1.0, 1.0, -1.0, -1.0]], np.float16)   # unit RMS
    wqn = np.array([2.0, 0.5, -1.0, 3.0])
    q, _, _ = orc.project_noise(h, P, P[:4], P[:4], wqn, np.ones(d), 0.0, nh, 1, d)
    want = (h[0, perm].astype(np.float64).reshape(nh, d)) * wqn
    np.testing.assert_allclose(q[0], want, rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------
# q8_0 blocks (Q1, Q2)
# ---------------------------------------------------------------------------

def test_q8_0_hand_values():
    """A block whose largest magnitude is 127 has scale 1: integer values are their own
    codes; 2.5 and -2.5 round away from zero; an all-zero block has scale 0; every block of
    32 has its own scale."""
    x = np.zeros(64)
    x[0], x[1], x[2], x[3], x[4] = 127.0, -127.0, 2.5, -2.5, 7.0
    x[32], x[33] = 0.5, -0.25                   # block 1: scale 0.5 / 127
    codes, scales = orc.q8_0_quantize(x)
    assert scales.dtype == np.float16 and codes.dtype == np.int8
    assert float(scales[0]) == 1.0
    assert list(codes[:5]) == [127, -127, 3, -3, 7] and not codes[5:32].any()
    assert float(scales[1]) == float(np.float16(np.float32(0.5) / np.float32(127)))
    assert list(codes[32:34]) == [127, -64] and not codes[34:].any()
    z_codes, z_scales = orc.q8_0_quantize(np.zeros(32))
    assert not z_codes.any() and float(z_scales[0]) == 0.0
    np.testing.assert_array_equal(orc.q8_0_dequantize(codes[:32], scales[:1]),
                                  [127, -127, 3, -3, 7] + [0] * 27)


def test_q8_0_error_bound_and_brute_force():
    """Round trip within half a step plus the F16 scale rounding, and the codes equal a
    plain per-element loop in float32."""
    rng = np.random.default_rng(8)
    x = rng.standard_normal((5, 128)) * np.array([1e-3, 1.0, 30.0, 0.2, 5.0])[:, None]
    codes, scales = orc.q8_0_quantize(x)
    back = orc.q8_0_dequantize(codes, scales)
    for r in range(5):
        for b in range(4):
            blk = x[r, 32 * b:32 * b + 32].astype(np.float32)
            d = np.float32(np.max(np.abs(blk))) / np.float32(127)
            inv = np.float32(1) / d
            for j in range(32):
                v = float(np.float32(blk[j] * inv))
                want = int(math.copysign(math.floor(abs(v) + 0.5), v))
                assert codes[r, 32 * b + j] == want
            # x' - x = (q d - x) + q (d_f16 - d): half a step plus the scale's rounding
            err = np.abs(back[r, 32 * b:32 * b + 32] - x[r, 32 * b:32 * b + 32])
            d16 = float(np.float16(d))
            bound = 0.5 * float(d) * (1 + 1e-6) + 127 * abs(d16 - float(d)) + 1e-30
            assert np.all(err <= bound)


def test_q8_0_ring_equals_dense():
    """O1 with q8_0 slots (K quantised after RoPE, V as given, noise rows too) equals O2
    with the same quantisation of exactly the window."""
    import synth
    import torch
    w = synth.workload(1, n_layer=1, swa_window=24)
    r = orc.RingOracle(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer, w.rope_theta,
                       swa_window=w.swa_window, kv_format="q8_0")
    for t, c in enumerate(synth.commit_schedule(w, 12)[:, 0]):
        c = int(c)
        start, _ = r.rows_needed(c)
        pos = torch.arange(start, c)
        k, v = synth.context_rows(w.seed, 0, 0, pos, w.kv_row, w.sigma)
        r.begin_step(c, k.numpy()[None], v.numpy()[None], start)
        q = synth.query_block(w.seed, t, 0, 0, w.q_len, w.n_head, w.head_dim, w.sigma).numpy()
        kn, vn = synth.noise_rows(w.seed, t, 0, 0, w.q_len, w.kv_row, w.sigma)
        for kind in ("full", "swa"):
            o1 = r.attend(0, q, kn.numpy(), vn.numpy(), kind)

            def rows(p):
                kk, vv = synth.context_rows(w.seed, 0, 0, torch.as_tensor(p), w.kv_row, w.sigma)
                return kk.numpy(), vv.numpy()
            o2 = orc.attend_dense(c, w.cap, rows, q, kn.numpy(), vn.numpy(), w.head_dim,
                                  w.n_head_kv, w.n_head, w.rope_theta, kind=kind,
                                  swa_window=w.swa_window, kv_format="q8_0")
            assert float(np.abs(o1 - o2).max()) < 1e-12
