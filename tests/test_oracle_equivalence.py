"""The ring oracle (O1) against the dense-window oracle (O2), the negative model of the
naive roll, and path independence of the bulk append.  CPU only.

The page "DFLASH2_RING_PORT.md" (section 1.7) states that the ring's result equals a
recompute over the full window; here the two oracles are built independently (the
ring keeps slots, the dense one regenerates rows by absolute position) and must agree
to float64 rounding.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import ring_oracle as orc


def _context_rows(w, seq, layer, pos):
    k, v = synth.context_rows(w.seed, seq, layer, torch.as_tensor(pos), w.kv_row, w.sigma)
    return k.numpy(), v.numpy()


def _produced_rows(hidden, eps):
    """Rows made by the context-row producer from seeded features and weights."""
    cache = {}

    def rows(w, seq, layer, pos):
        if layer not in cache:
            cache[layer] = [x.numpy() for x in synth.producer_weights(w.seed, layer, w.kv_row,
                                                                      hidden, w.head_dim)]
        wk, wv, kn = cache[layer]
        feat = synth.feature_rows(w.seed, seq, torch.as_tensor(pos, dtype=torch.int64), hidden,
                                  w.sigma).numpy()
        return orc.produce_rows(feat, wk, wv, kn, eps, w.n_head_kv, w.head_dim)
    return rows


def _rows_fn(w, seq, layer, source=_context_rows):
    return lambda pos: source(w, seq, layer, np.asarray(pos))


def _step_rows(w, seq, start, c, source=_context_rows):
    pos = np.arange(start, c)
    ks, vs = [], []
    for layer in range(w.n_layer):
        k, v = source(w, seq, layer, pos)
        ks.append(k)
        vs.append(v)
    return np.stack(ks), np.stack(vs)


def _run_equivalence(w, n_steps, kinds, source=_context_rows, kv_format="f16"):
    r = orc.RingOracle(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer,
                       w.rope_theta, swa_window=w.swa_window, kv_format=kv_format)
    sched = synth.commit_schedule(w, n_steps)
    worst = 0.0
    for t, c in enumerate(sched[:, 0]):
        c = int(c)
        start, _ = r.rows_needed(c)
        k, v = _step_rows(w, 0, start, c, source)
        r.begin_step(c, k, v, start)
        for layer in range(w.n_layer):
            q = synth.query_block(w.seed, t, 0, layer, w.q_len, w.n_head, w.head_dim, w.sigma)
            kn, vn = synth.noise_rows(w.seed, t, 0, layer, w.q_len, w.kv_row, w.sigma)
            for kind in kinds:
                o1 = r.attend(layer, q.numpy(), kn.numpy(), vn.numpy(), kind)
                o2 = orc.attend_dense(c, w.cap, _rows_fn(w, 0, layer, source), q.numpy(), kn.numpy(),
                                      vn.numpy(), w.head_dim, w.n_head_kv, w.n_head,
                                      w.rope_theta, kind=kind, swa_window=w.swa_window,
                                      kv_format=kv_format)
                worst = max(worst, float(np.abs(o1 - o2).max()))
    return worst


def test_ring_equals_dense_window_tiny_workload():
    w = synth.workload(1, swa_window=24)            # cap 64, 40 steps, wraps ~3 times
    assert _run_equivalence(w, 40, ("full", "swa")) < 1e-12


def test_ring_equals_dense_window_with_bulk_jumps():
    w = synth.workload(3, cap=48, n_layer=2, head_dim=16, n_head_kv=2, n_head=4,
                       extra={"jump_max": 400, "fold_max": 18, "p_jump": 0.4})
    assert _run_equivalence(w, 30, ("full",)) < 1e-12


def test_ring_equals_dense_window_with_produced_rows():
    """The same equivalence when the context rows come from the producer (P1-P3)."""
    w = synth.workload(3, cap=48, n_layer=2, head_dim=16, n_head_kv=2, n_head=4,
                       extra={"jump_max": 200, "fold_max": 18, "p_jump": 0.3})
    assert _run_equivalence(w, 20, ("full",), _produced_rows(64, 1e-6)) < 1e-12


def test_q8_0_ring_equals_dense_window_with_produced_rows_and_jumps():
    """q8_0 slots (Q1, Q2) with rows from the producer, bulk jumps past the ring and both
    masks: the ring's state-by-step route and the dense route quantise the same rows the
    same way, so they agree to float64 rounding."""
    w = synth.workload(3, cap=64, n_layer=2, head_dim=32, n_head_kv=2, n_head=4, swa_window=20,
                       extra={"jump_max": 300, "fold_max": 18, "p_jump": 0.3})
    assert _run_equivalence(w, 16, ("full", "swa"), _produced_rows(64, 1e-6), "q8_0") < 1e-12


def test_naive_roll_differs_once_rows_are_evicted():
    """Negative model (section 2.2): a cache of cap cells without a window mask agrees
    with the ring while nothing is evicted and departs from it afterwards."""
    w = synth.workload(1, head_dim=16, n_head_kv=2, n_head=4)
    r = orc.RingOracle(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, 1, w.rope_theta)
    naive = orc.NaiveRollOracle(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head,
                                w.rope_theta)
    agreed_before, differed_after = False, False
    for t, c in enumerate(synth.commit_schedule(w, 40)[:, 0]):
        c = int(c)
        prev = naive.next_pos
        k, v = _step_rows(w, 0, prev, c)
        start, _ = r.rows_needed(c)
        r.begin_step(c, k[:, start - prev:], v[:, start - prev:], start)
        naive.begin_step(c, k[0], v[0], prev)
        q = synth.query_block(w.seed, t, 0, 0, w.q_len, w.n_head, w.head_dim, w.sigma).numpy()
        kn, vn = [x.numpy() for x in synth.noise_rows(w.seed, t, 0, 0, w.q_len, w.kv_row, w.sigma)]
        o_ring = r.attend(0, q, kn, vn, "full")
        o_naive = naive.attend(q, kn, vn)
        err = float(np.abs(o_ring - o_naive).max())
        if c + w.q_len <= w.cap:
            assert err < 1e-12
            agreed_before = True
        elif c > w.cap + w.q_len:
            differed_after = differed_after or err > 1e-2
    assert agreed_before and differed_after


def test_bulk_chunking_and_prefill_route_do_not_change_state():
    """Chunk size of the bulk path, and one prefill vs several, leave the same state."""
    w = synth.workload(2, cap=256, n_layer=2, head_dim=16, n_head_kv=2, n_head=4)
    args = (w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer, w.rope_theta)
    k, v = _step_rows(w, 0, 0, 512)
    a = orc.RingOracle(*args, bulk_chunk=1024)
    a.begin_step(512, k[:, 256:], v[:, 256:], 256)
    b = orc.RingOracle(*args, bulk_chunk=7)
    b.begin_step(512, k[:, 256:], v[:, 256:], 256)
    c = orc.RingOracle(*args, bulk_chunk=64)
    for cc in (64, 128, 192, 256, 320, 384, 448, 512):
        st, _ = c.rows_needed(cc)
        c.begin_step(cc, k[:, st:cc], v[:, st:cc], st)
    for other in (b, c):
        np.testing.assert_array_equal(a.slot_pos, other.slot_pos)
        np.testing.assert_array_equal(a.k[:, :w.cap], other.k[:, :w.cap])
        np.testing.assert_array_equal(a.v[:, :w.cap], other.v[:, :w.cap])
        np.testing.assert_array_equal(a.mask_full(), other.mask_full())
    assert a.last_path == "bulk"


@pytest.mark.parametrize("seq", [0, 3])
def test_generator_rows_are_pure_functions_of_position(seq):
    w = synth.workload(4)
    k1, v1 = synth.context_rows(w.seed, seq, 2, torch.tensor([5, 131071, 77]), w.kv_row, w.sigma)
    k2, v2 = synth.context_rows(w.seed, seq, 2, torch.tensor([77, 5]), w.kv_row, w.sigma)
    assert torch.equal(k1[0], k2[1]) and torch.equal(k1[2], k2[0])
    assert torch.equal(v1[0], v2[1])
    assert not torch.equal(k1[0], v1[0])
