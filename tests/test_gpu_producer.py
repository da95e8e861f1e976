"""Parity of the context-row producer (ring_begin_step_features) with the float64 oracle.

The CUDA path projects seeded fused features with seeded weights on the tensor cores,
normalises K per head, turns it by RoPE and writes both rows into the ring; the oracle
does the same in float64 (readings P1-P3 of oracle/ring_oracle.py) and is fed the same
features and weights, drawn on the CPU by the same counter-based generator.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import ring_oracle as orc
from speculative_decoding_draft_kv_gb300 import ring as R
from tests.ring_harness import (ATOL, REL_L2, assert_close, expected_tile_flags, f16_spacing,
                                f16_within, projection_error_bound, rel_l2)

pytestmark = pytest.mark.gpu

EPS = 1e-6


class ProducerRun:
    """A CUDA ring fed by the producer, plus per-sequence bookkeeping oracles."""

    def __init__(self, w, hidden, swa_window=None, tiles_per_split=0, kv_format="f16"):
        self.w, self.hidden = w, hidden
        self.kv_format = kv_format
        self.swa = w.swa_window if swa_window is None else swa_window
        self.dev = torch.device("cuda")
        self.ring = R.Ring(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer,
                           w.rope_theta, n_seq=w.n_seq, swa_window=self.swa,
                           tiles_per_split=tiles_per_split, kv_format=kv_format)
        self.g = self.ring.geometry
        cpu = [synth.producer_weights(w.seed, l, w.kv_row, hidden, w.head_dim)
               for l in range(w.n_layer)]
        self.wk = [x[0].numpy() for x in cpu]
        self.wv = [x[1].numpy() for x in cpu]
        self.kn = [x[2].numpy() for x in cpu]
        gpu = [synth.producer_weights(w.seed, l, w.kv_row, hidden, w.head_dim, device=self.dev)
               for l in range(w.n_layer)]
        self.gwk = torch.stack([x[0] for x in gpu]).contiguous()
        self.gwv = torch.stack([x[1] for x in gpu]).contiguous()
        self.gkn = torch.stack([x[2] for x in gpu]).contiguous()
        self.ring.set_producer(hidden, EPS, self.gwk, self.gwv, self.gkn)
        self.book = [orc.RingOracle(w.cap, w.q_len, 2, 1, 1, 1, w.rope_theta,
                                    swa_window=self.swa) for _ in range(w.n_seq)]
        self.committed = np.zeros(w.n_seq, np.int64)
        self._keep = None

    def close(self):
        self.ring.close()

    def feat(self, seq, pos):
        return synth.feature_rows(self.w.seed, seq, torch.as_tensor(np.asarray(pos, np.int64)),
                                  self.hidden, self.w.sigma).numpy()

    def rows(self, seq, layer, pos):
        """Oracle rows (pre-RoPE K float64, V F16) of positions ``pos``."""
        return orc.produce_rows(self.feat(seq, pos), self.wk[layer], self.wv[layer],
                                self.kn[layer], EPS, self.w.n_head_kv, self.w.head_dim)

    def begin_step(self, committed, recompute=False):
        """``recompute``: the legacy path -- every row of [lo, c) produced again."""
        w = self.w
        committed = np.asarray(committed, np.int64)
        starts, counts = [], []
        for s in range(w.n_seq):
            st, nn = self.book[s].rows_needed(int(committed[s]))
            if recompute:
                c = int(committed[s])
                st, nn = c - min(c, w.cap), min(c, w.cap)
            starts.append(st)
            counts.append(nn)
        n_rows = int(sum(counts))
        row_off = np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int64)
        feat = None
        if n_rows:
            feat = torch.empty((n_rows, self.hidden), dtype=torch.float16, device=self.dev)
            for s in range(w.n_seq):
                if counts[s]:
                    a = int(row_off[s])
                    feat[a:a + counts[s]] = synth.feature_rows(
                        w.seed, s, torch.arange(starts[s], committed[s], device=self.dev),
                        self.hidden, w.sigma, device=self.dev)
        step = self.ring.recompute_window if recompute else self.ring.begin_step_features
        step(committed, feat, row_off, np.asarray(starts, np.int64))
        self._keep = feat
        paths = []
        for s in range(w.n_seq):
            st, nn = self.book[s].rows_needed(int(committed[s]))
            z = np.zeros((1, nn, 2), np.float16)
            paths.append(self.book[s].begin_step(int(committed[s]), z, z, st))
        self.committed = committed.copy()
        return paths

    def check_state(self, seqs=None):
        for s in (range(self.w.n_seq) if seqs is None else seqs):
            b = self.book[s]
            np.testing.assert_array_equal(self.ring.slot_pos(s), b.slot_pos.astype(np.int32))
            for kind in ["full"] + (["swa"] if self.swa else []):
                want = b.mask(kind)
                assert self.ring.mask(s, kind).view(np.uint32).tobytes() == \
                    want.view(np.uint32).tobytes(), (s, kind)
                np.testing.assert_array_equal(self.ring.tile_flags(s, kind),
                                              expected_tile_flags(want, self.g["tile_slots"]))

    def check_kv(self, seq, layer, slots=None):
        """K and V of (sampled) filled slots against the oracle's produced rows."""
        sp = self.book[seq].slot_pos
        slots = np.flatnonzero(sp >= 0) if slots is None else np.asarray(
            [s for s in slots if sp[s] >= 0], np.int64)
        if self.kv_format == "q8_0":
            return self.check_kv_q8(seq, layer, slots)
        k, v = self.ring.kv(seq, layer)
        if not len(slots):
            return
        pos = sp[slots]
        w, hd, nh = self.w, self.w.head_dim, self.w.n_head_kv
        x = self.feat(seq, pos)
        v_exact = x @ self.wv[layer].astype(np.float64).T
        # V: the F16 rounding of a float32 accumulation of exact products
        assert f16_within(v[slots], v_exact, projection_error_bound(x, self.wv[layer])), layer
        k_exact, bound = self.k_exact_and_bound(x, pos, layer)
        assert f16_within(k[slots], k_exact, bound), layer
        t = self.g["trash_slot"]
        assert np.all(k[t] == 0) and np.all(v[t] == 0)

    def k_exact_and_bound(self, x, pos, layer):
        """Exact rotated K rows of features x and the bound on the GPU's float32 value."""
        w, hd, nh = self.w, self.w.head_dim, self.w.n_head_kv
        k_pre = x @ self.wk[layer].astype(np.float64).T
        # K: the accumulation error carried through the per-head norm and the rotation:
        # e = |dk| / rms + |k| |drms| / rms^2 per element with |drms| <= max |dk| of the
        # head, times max |w|, and a rotation adds two such errors; the float32 norm and
        # RoPE (cos/sin within 2 float32 units, products and FMAs rounded once each) add
        # at most 5e-7 (|y1| + |y2|) <= 1.2e-6 max |y| of the head.
        dk = projection_error_bound(x, self.wk[layer]).reshape(len(pos), nh, hd)
        kh = k_pre.reshape(len(pos), nh, hd)
        rms = np.sqrt(np.mean(kh * kh, axis=-1, keepdims=True) + EPS)
        e = (dk + np.abs(kh) * dk.max(axis=-1, keepdims=True) / rms) / rms
        y = orc.rms_norm_heads(k_pre, self.kn[layer], EPS, nh, hd)
        ymax = np.abs(y.reshape(len(pos), nh, hd)).max(axis=-1, keepdims=True)
        e = 2.0 * e.max(axis=-1, keepdims=True) * np.abs(self.kn[layer]).max() + 1.2e-6 * ymax + 1e-7
        k_exact = orc.rope_rows(y, pos, nh, hd, w.rope_theta)
        bound = np.broadcast_to(e, kh.shape).reshape(len(pos), nh * hd)
        return k_exact, bound

    def check_kv_q8(self, seq, layer, slots):
        """q8_0 slots: each read-back value code * scale within its quantisation error of
        the exact row plus the GPU's own error before quantising.  The GPU decides
        d = max|x| / 127 and codes round(x / d) on its float32 value x (K straight from the
        rotation, V after its F16 rounding) and stores d as F16, so |code * d16 - exact| <=
        d / 2 + 127 |d16 - d| + |x - exact|, with d <= d16 + ulp(d16) / 2."""
        kc, ks, vc, vs = self.ring.kv_q8(seq, layer)
        t = self.g["trash_slot"]
        assert not kc[t].any() and not vc[t].any()
        assert not ks[t].view(np.uint16).any() and not vs[t].view(np.uint16).any()
        if not len(slots):
            return
        pos = self.book[seq].slot_pos[slots]
        x = self.feat(seq, pos)

        def read_back(codes, scales):
            sc = np.repeat(scales.astype(np.float64), orc.Q8_BLOCK, axis=-1)
            u = np.repeat(f16_spacing(scales.astype(np.float64)), orc.Q8_BLOCK, axis=-1)
            return codes.astype(np.float64) * sc, 0.5 * (sc + 0.5 * u) * (1 + 1e-4) + 63.5 * u

        v_exact = x @ self.wv[layer].astype(np.float64).T
        pv = projection_error_bound(x, self.wv[layer])
        got, qb = read_back(vc[slots], vs[slots])
        ev = pv + f16_spacing(np.abs(v_exact) + pv)
        assert np.all(np.abs(got - v_exact) <= qb + ev + 1e-12), layer
        k_exact, bound = self.k_exact_and_bound(x, pos, layer)
        got, qb = read_back(kc[slots], ks[slots])
        assert np.all(np.abs(got - k_exact) <= qb + bound + 1e-12), layer

    def attend(self, step, layer, kind):
        w = self.w
        qs, ks, vs = [], [], []
        for s in range(w.n_seq):
            qs.append(synth.query_block(w.seed, step, s, layer, w.q_len, w.n_head, w.head_dim,
                                        w.sigma, device=self.dev))
            kk, vv = synth.noise_rows(w.seed, step, s, layer, w.q_len, w.kv_row, w.sigma,
                                      device=self.dev)
            ks.append(kk)
            vs.append(vv)
        q, kn, vn = torch.stack(qs), torch.stack(ks), torch.stack(vs)
        o = torch.empty_like(q)
        self.ring.attend(layer, kind, q, kn, vn, o)
        torch.cuda.synchronize()
        return o.cpu().numpy()

    def expected(self, step, layer, kind, seq, heads=None):
        w = self.w
        q = synth.query_block(w.seed, step, seq, layer, w.q_len, w.n_head, w.head_dim, w.sigma)
        kn, vn = synth.noise_rows(w.seed, step, seq, layer, w.q_len, w.kv_row, w.sigma)
        return orc.attend_dense(int(self.committed[seq]), w.cap,
                                lambda pos: self.rows(seq, layer, pos), q.numpy(), kn.numpy(),
                                vn.numpy(), w.head_dim, w.n_head_kv, w.n_head, w.rope_theta,
                                kind=kind, swa_window=self.swa, heads=heads,
                                kv_format=self.kv_format)

    def q8_bound(self, seq, layer, q, k_noise, v_noise, kind):
        """Elementwise allowance [q_len, n_head, head_dim] for attention over q8_0 rows made
        on the GPU, from the codes that actually differ.  The GPU quantises its float32
        rows and the oracle its float64 rows, so where the two straddle a rounding boundary
        a code differs by one, and a block maximum -- its scale -- by one F16 step (the slot
        checks bound both).  Only the slots of this attention matter: their read-back
        values on both sides give |dK| and |dV| per element.  Through the oracle's own
        float64 softmax weights p: a value moved by dV moves the output by p * dV; a key
        moved by dK moves its logit by scale * |q| . |dK| = delta and the output by at
        most p * delta * 2 max|v| (times exp(2 max delta) for the second order).  The GPU's
        rows serve only this tolerance; the expected output is the oracle's alone."""
        w, c = self.w, int(self.committed[seq])
        win = min(c, w.cap)
        lo = c - (min(self.swa, win) if kind == "swa" else win)
        pos = np.arange(lo, c, dtype=np.int64)
        k_pre, v = self.rows(seq, layer, pos)
        k_rot = orc.rope_rows(np.asarray(k_pre, np.float64), pos, w.n_head_kv, w.head_dim, w.rope_theta)
        kn_rot = orc.rope_rows(np.asarray(k_noise, np.float64), c + np.arange(w.q_len), w.n_head_kv,
                               w.head_dim, w.rope_theta)
        k_or = orc.q8_0_round_trip(np.concatenate([k_rot, kn_rot]))
        v_or = orc.q8_0_round_trip(np.concatenate([np.asarray(v, np.float64), np.asarray(v_noise, np.float64)]))
        kc, ks, vc, vs = self.ring.kv_q8(seq, layer)
        slots = np.concatenate([pos % w.cap, w.cap + np.arange(w.q_len)])
        k_gpu = orc.q8_0_dequantize(kc[slots], ks[slots])
        v_gpu = orc.q8_0_dequantize(vc[slots], vs[slots])
        dk, dv = np.abs(k_gpu - k_or), np.abs(v_gpu - v_or)
        n_ctx = len(pos)
        mask = np.zeros((w.q_len, n_ctx + w.q_len))
        if kind == "swa":
            mask[:, n_ctx:] = np.where(np.arange(w.q_len)[None, :] > np.arange(w.q_len)[:, None], -np.inf, 0.0)
        qr = orc.rope_neox(np.asarray(q, np.float64), (c + np.arange(w.q_len))[:, None], w.rope_theta)
        scale = 1.0 / np.sqrt(w.head_dim)
        G, d = w.n_head // w.n_head_kv, w.head_dim
        vmax = max(float(np.abs(v_or).max()), float(np.abs(v_gpu).max()))
        bound = np.zeros((w.q_len, w.n_head, d))
        for h in range(w.n_head):
            g = h // G
            kh, dkh, dvh = k_or[:, g * d:(g + 1) * d], dk[:, g * d:(g + 1) * d], dv[:, g * d:(g + 1) * d]
            sc = qr[:, h] @ kh.T * scale + mask
            p = np.exp(sc - sc.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            delta = scale * (np.abs(qr[:, h]) @ dkh.T)                # [q_len, keys]
            second = np.exp(2.0 * float(delta.max(initial=0.0)))
            bound[:, h] = (p @ dvh + 2.0 * vmax * (p * delta).sum(axis=1)[:, None]) * second
        return bound


def assert_close_q8(got, want, bound, what=""):
    """The attention bar (max-abs 2e-3, relative L2 1e-3) with max-abs widened, element by
    element, by the allowance of the codes that differ between the two quantisations
    (q8_bound); relative L2 unchanged.  The widening must stay below 2 x 2e-3."""
    err = np.abs(got - want)
    rl2 = rel_l2(got, want)
    extra = float(np.max(bound, initial=0.0))
    assert extra <= 2 * ATOL, f"{what}: allowance {extra:.3g} above twice the bar"
    assert np.all(err <= ATOL + bound) and rl2 <= REL_L2, \
        f"{what}: max abs {err.max():.3g} (allowance up to {extra:.3g}), rel L2 {rl2:.3g}"
    return extra


def test_feature_and_weight_generators_bit_identical_on_gpu():
    dev = torch.device("cuda")
    a = synth.feature_rows(3, 1, torch.arange(100, 140), 512, 0.5)
    b = synth.feature_rows(3, 1, torch.arange(100, 140, device=dev), 512, 0.5, device=dev)
    assert torch.equal(a, b.cpu())
    for x, y in zip(synth.producer_weights(3, 2, 256, 512, 128),
                    synth.producer_weights(3, 2, 256, 512, 128, device=dev)):
        assert torch.equal(x, y.cpu())


@pytest.mark.parametrize("hidden", [256, 320])
def test_small_rings_full_state(hidden):
    """Two sequences, fold-in and bulk steps (and a jump past the ring), every slot of
    every layer checked, both masks, attention against the dense window of produced rows.
    hidden 320 splits unevenly over the cluster (5 stages of 64)."""
    w = synth.workload(1, n_layer=2, n_seq=2, swa_window=24)
    run = ProducerRun(w, hidden)
    try:
        sched = [[5, 0], [12, 9], [40, 30], [41, 200], [60, 207], [140, 215], [149, 216]]
        for t, c in enumerate(sched):
            run.begin_step(c)
            run.check_state()
            for s in range(w.n_seq):
                for layer in range(w.n_layer):
                    run.check_kv(s, layer)
            for kind in ("full", "swa"):
                layer = t % 2
                o = run.attend(t, layer, kind)
                for s in range(w.n_seq):
                    assert_close(o[s], run.expected(t, layer, kind, s), f"step {t} seq {s} {kind}")
        assert run.ring.device_error() == 0
    finally:
        run.close()


@pytest.mark.parametrize("hidden,kv_format", [(256, "f16"), (320, "f16"), (256, "q8_0")])
def test_many_rows_on_the_tensor_core_path(hidden, kv_format):
    """Steps of 256 rows and more in one contiguous run of features go to the tcgen05
    kernel (128-row tiles, accumulators in tensor memory): a partial last tile, two
    sequences packed in one run, a whole-ring jump; every slot of every layer against the
    float64 oracle within the float32-accumulation bound, state bit-exact, attention."""
    w = synth.workload(1, cap=1024, n_layer=2, n_seq=2, swa_window=300)
    run = ProducerRun(w, hidden, kv_format=kv_format)
    try:
        for t, c in enumerate([[300, 0], [301, 500], [1400, 700], [1401, 2900]]):
            run.begin_step(c)
            run.check_state()
            for s in range(w.n_seq):
                for layer in range(w.n_layer):
                    run.check_kv(s, layer)
            if kv_format == "f16":
                o = run.attend(t, t % 2, "full")
                for s in range(w.n_seq):
                    assert_close(o[s], run.expected(t, t % 2, "full", s), f"step {t} seq {s}")
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_steady_decode_full_size():
    """cap 4096, 5 layers, hidden 4096: an 8192-row prefill (bulk) then decode steps of
    the acceptance histogram; sampled slots of every layer and sampled heads of the
    attention output."""
    w = synth.workload(2)
    run = ProducerRun(w, 4096)
    rng = np.random.default_rng(1)
    try:
        sched = synth.commit_schedule(w, 4)
        for t, c in enumerate(sched):
            run.begin_step(c)
            run.check_state()
            lo = int(c[0]) - min(int(c[0]), w.cap)
            recent = [int(p) % w.cap for p in range(max(lo, int(c[0]) - 9), int(c[0]))]
            slots = sorted(set(rng.integers(0, w.cap, 24).tolist() + recent))
            for layer in (0, 4):
                run.check_kv(0, layer, slots)
            heads = [0, 13, 31]
            layer = t % w.n_layer
            o = run.attend(t, layer, "full")
            want = run.expected(t, layer, "full", 0, heads=heads)
            assert_close(o[0][:, heads], want[:, heads], f"step {t}")
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_producer_errors_and_state_unchanged():
    w = synth.workload(1, n_layer=2)
    ring = R.Ring(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer, w.rope_theta)
    dev = torch.device("cuda")
    try:
        feat = torch.zeros((4, 256), dtype=torch.float16, device=dev)
        with pytest.raises(R.RingError) as e:               # no producer yet
            ring.begin_step_features([4], feat, [0], [0])
        assert e.value.code == R.RING_ESTATE
        wk = torch.zeros((2, w.kv_row, 256), dtype=torch.float16, device=dev)
        kn = torch.ones((2, w.head_dim), dtype=torch.float32, device=dev)
        with pytest.raises(R.RingError) as e:               # hidden not a multiple of 64
            ring.set_producer(200, EPS, wk, wk, kn)
        assert e.value.code == R.RING_EINVAL
        ring.set_producer(256, EPS, wk, wk, kn)
        with pytest.raises(R.RingError) as e:               # rows do not cover [start, c)
            ring.begin_step_features([10], feat, [0], [0])
        assert e.value.code == R.RING_ERANGE
        np.testing.assert_array_equal(ring.slot_pos(), np.full(w.cap, -1, np.int32))
        ring.begin_step_features([4], feat, [0], [0])      # zero weights: K and V rows of 0
        torch.cuda.synchronize()
        np.testing.assert_array_equal(ring.slot_pos()[:4], [0, 1, 2, 3])
        k, v = ring.kv(0, 1)
        assert np.all(k[:4] == 0) and np.all(v[:4] == 0)
        assert ring.device_error() == 0
        ring.set_producer(None, 0.0, None, None, None)      # detached again
        with pytest.raises(R.RingError) as e:
            ring.begin_step_features([8], feat, [0], [4])
        assert e.value.code == R.RING_ESTATE
    finally:
        ring.close()


def test_many_sequences_read_the_staged_step_state():
    """More sequences than travel as kernel parameters: the producer reads the row ranges
    from the staged step state instead."""
    w = synth.workload(1, n_layer=1, n_seq=20)
    run = ProducerRun(w, 128)
    try:
        rng = np.random.default_rng(4)
        c = np.zeros(w.n_seq, np.int64)
        for t in range(3):
            c = c + rng.integers(0, 40, w.n_seq)
            run.begin_step(c)
            run.check_state()
            for s in range(w.n_seq):
                run.check_kv(s, 0)
            o = run.attend(t, 0, "full")
            for s in (0, 7, 19):
                assert_close(o[s], run.expected(t, 0, "full", s), f"step {t} seq {s}")
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_legacy_window_recompute_equals_the_ring():
    """The page's legacy path (the whole window produced again every step) leaves the
    same ring state and gives the same attention as the ring's incremental appends."""
    w = synth.workload(1, n_layer=2, n_seq=2, swa_window=24)
    run = ProducerRun(w, 192)
    try:
        for t, c in enumerate([[5, 3], [30, 12], [90, 70], [95, 75], [300, 76]]):
            run.begin_step(c, recompute=True)
            run.check_state()
            for s in range(w.n_seq):
                for layer in range(w.n_layer):
                    run.check_kv(s, layer)
            for kind in ("full", "swa"):
                o = run.attend(t, t % 2, kind)
                for s in range(w.n_seq):
                    assert_close(o[s], run.expected(t, t % 2, kind, s), f"step {t} seq {s} {kind}")
        assert run.ring.device_error() == 0
    finally:
        run.close()


class DraftRun(ProducerRun):
    """ProducerRun plus the query projection, for ring_draft_step."""

    def __init__(self, w, hidden, pattern, kv_format="f16"):
        super().__init__(w, hidden, kv_format=kv_format)
        self.pattern = pattern
        qw = [synth.query_weights(w.seed, l, w.n_head * w.head_dim, hidden, w.head_dim)
              for l in range(w.n_layer)]
        self.wq = [x[0].numpy() for x in qw]
        self.qn = [x[1].numpy() for x in qw]
        gq = [synth.query_weights(w.seed, l, w.n_head * w.head_dim, hidden, w.head_dim,
                                  device=self.dev) for l in range(w.n_layer)]
        self.gwq = torch.stack([x[0] for x in gq]).contiguous()
        self.gqn = torch.stack([x[1] for x in gq]).contiguous()
        self.ring.set_producer(hidden, EPS, self.gwk, self.gwv, self.gkn, self.gwq, self.gqn)

    def step(self, t, committed):
        """One ring_draft_step; returns the outputs [n_layer] as numpy arrays."""
        w = self.w
        committed = np.asarray(committed, np.int64)
        starts, counts = [], []
        for s in range(w.n_seq):
            st, nn = self.book[s].rows_needed(int(committed[s]))
            starts.append(st)
            counts.append(nn)
        n_rows = int(sum(counts))
        row_off = np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int64)
        feat = None
        if n_rows:
            feat = torch.empty((n_rows, self.hidden), dtype=torch.float16, device=self.dev)
            for s in range(w.n_seq):
                if counts[s]:
                    a = int(row_off[s])
                    feat[a:a + counts[s]] = synth.feature_rows(
                        w.seed, s, torch.arange(starts[s], committed[s], device=self.dev),
                        self.hidden, w.sigma, device=self.dev)
        h = torch.stack([torch.stack([synth.noise_hidden(w.seed, t, s, l, w.q_len, self.hidden,
                                                         w.sigma, device=self.dev)
                                      for s in range(w.n_seq)]) for l in range(w.n_layer)])
        o = [torch.empty((w.n_seq, w.q_len, w.n_head, w.head_dim), device=self.dev)
             for _ in range(w.n_layer)]
        self.ring.draft_step(committed, feat, row_off, np.asarray(starts, np.int64),
                             h.contiguous(), self.pattern, o)
        torch.cuda.synchronize()
        for s in range(w.n_seq):
            z = np.zeros((1, counts[s], 2), np.float16)
            self.book[s].begin_step(int(committed[s]), z, z, starts[s])
        self.committed = committed.copy()
        return [x.cpu().numpy() for x in o]

    def noise_qkv(self, t, layer, seq):
        w = self.w
        h = synth.noise_hidden(w.seed, t, seq, layer, w.q_len, self.hidden, w.sigma).numpy()
        return orc.project_noise(h, self.wq[layer], self.wk[layer], self.wv[layer],
                                 self.qn[layer], self.kn[layer], EPS, w.n_head,
                                 w.n_head_kv, w.head_dim)

    def draft_bound(self, t, layer, seq):
        q, kn, vn = self.noise_qkv(t, layer, seq)
        return self.q8_bound(seq, layer, q, kn, vn, self.pattern[layer])

    def expected_draft(self, t, layer, seq, heads=None):
        w = self.w
        q, kn, vn = self.noise_qkv(t, layer, seq)
        return orc.attend_dense(int(self.committed[seq]), w.cap,
                                lambda pos: self.rows(seq, layer, pos), q, kn, vn, w.head_dim,
                                w.n_head_kv, w.n_head, w.rope_theta, kind=self.pattern[layer],
                                swa_window=self.swa, heads=heads, kv_format=self.kv_format)


def test_draft_step_small_rings_mixed_pattern():
    """ring_draft_step: context rows from features, noise Q/K/V from each layer's hidden
    states, a full / SWA / full layer pattern; every output against the float64 route."""
    w = synth.workload(1, n_layer=3, n_seq=2, swa_window=24)
    run = DraftRun(w, 192, ["full", "swa", "full"])
    try:
        for t, c in enumerate([[5, 0], [14, 9], [60, 41], [63, 200], [150, 205]]):
            outs = run.step(t, c)
            run.check_state()
            for layer in range(w.n_layer):
                for s in range(w.n_seq):
                    assert_close(outs[layer][s], run.expected_draft(t, layer, s),
                                 f"step {t} layer {layer} seq {s}")
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_draft_step_kernel_clock_counts_each_kind():
    """The device clock keeps one span per launch and kind through ring_draft_step: the
    context-row producer once per step with new rows, the noise projections and the
    attention once per layer; each kind's time fits inside the steps' event time, and the
    outputs stay those of the float64 route."""
    w = synth.workload(1, n_layer=3, n_seq=2, swa_window=24)
    run = DraftRun(w, 192, ["full", "swa", "full"])
    try:
        run.step(0, [5, 0])
        run.ring.clock_enable(True)
        for kind in ("attend", "produce", "project"):
            assert run.ring.clock_read(kind) == (0.0, 0)
        steps = [[14, 9], [60, 41], [63, 200], [63, 200], [150, 205]]
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        outs = [run.step(1 + t, c) for t, c in enumerate(steps)]
        b.record()
        torch.cuda.synchronize()
        ev_ms = a.elapsed_time(b)
        got = {kind: run.ring.clock_read(kind) for kind in ("attend", "produce", "project")}
        prev = [[5, 0]] + steps[:-1]
        with_rows = sum(1 for c, p in zip(steps, prev) if c != p)   # no rows: no producer launch
        assert got["produce"][1] == with_rows
        assert got["project"][1] == w.n_layer * len(steps)
        assert got["attend"][1] == w.n_layer * len(steps)
        for kind, (ms, n) in got.items():
            assert 0.0 < ms <= ev_ms, kind
        t = len(steps)
        for layer in range(w.n_layer):
            for s in range(w.n_seq):
                assert_close(outs[-1][layer][s], run.expected_draft(t, layer, s),
                             f"step {t} layer {layer} seq {s}")
        assert R.library().ring_clock_read(run.ring.h, 3, None, None) == R.RING_EINVAL
        run.ring.clock_enable(False)
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_draft_step_full_size():
    """cap 4096, 5 layers, hidden 4096: prefill then decode steps, sampled heads."""
    w = synth.workload(2)
    run = DraftRun(w, 4096, ["full"] * w.n_layer)
    try:
        heads = [0, 17, 31]
        for t, c in enumerate(synth.commit_schedule(w, 2)):
            outs = run.step(t, c)
            for layer in (0, 4):
                want = run.expected_draft(t, layer, 0, heads=heads)
                assert_close(outs[layer][0][:, heads], want[:, heads], f"step {t} layer {layer}")
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_draft_step_needs_query_weights():
    w = synth.workload(1, n_layer=1)
    run = ProducerRun(w, 128)
    try:
        h = torch.zeros((1, 1, w.q_len, 128), dtype=torch.float16, device=run.dev)
        o = [torch.empty((1, w.q_len, w.n_head, w.head_dim), device=run.dev)]
        with pytest.raises(R.RingError) as e:
            run.ring.draft_step([0], None, [0], [0], h, ["full"], o)
        assert e.value.code == R.RING_ESTATE
    finally:
        run.close()


def test_q8_small_rings_full_state():
    """q8_0 rings fed by the producer: two sequences, fold-in, bulk and a jump past the
    ring; every filled slot of every layer within its derived bound, both masks, and
    attention against the dense window of the oracle's produced rows, quantised."""
    w = synth.workload(1, n_layer=2, n_seq=2, swa_window=24)
    run = ProducerRun(w, 256, kv_format="q8_0")
    try:
        sched = [[5, 0], [12, 9], [40, 30], [41, 200], [60, 207], [140, 215], [149, 216]]
        for t, c in enumerate(sched):
            run.begin_step(c)
            run.check_state()
            for s in range(w.n_seq):
                for layer in range(w.n_layer):
                    run.check_kv(s, layer)
            for kind in ("full", "swa"):
                layer = t % 2
                o = run.attend(t, layer, kind)
                for s in range(w.n_seq):
                    q = synth.query_block(w.seed, t, s, layer, w.q_len, w.n_head, w.head_dim, w.sigma)
                    kn, vn = synth.noise_rows(w.seed, t, s, layer, w.q_len, w.kv_row, w.sigma)
                    bound = run.q8_bound(s, layer, q.numpy(), kn.numpy(), vn.numpy(), kind)
                    assert_close_q8(o[s], run.expected(t, layer, kind, s), bound,
                                    f"step {t} seq {s} {kind}")
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_q8_draft_step_small_rings_mixed_pattern():
    """ring_draft_step on q8_0 rings (context rows quantised by the producer, noise rows by
    the attention), a full / SWA / full pattern; every output against the float64 route."""
    w = synth.workload(1, n_layer=3, n_seq=2, swa_window=24)
    run = DraftRun(w, 192, ["full", "swa", "full"], kv_format="q8_0")
    try:
        for t, c in enumerate([[5, 0], [14, 9], [60, 41], [63, 200], [150, 205]]):
            outs = run.step(t, c)
            run.check_state()
            for s in range(w.n_seq):
                run.check_kv(s, t % w.n_layer)
            for layer in range(w.n_layer):
                for s in range(w.n_seq):
                    assert_close_q8(outs[layer][s], run.expected_draft(t, layer, s),
                                    run.draft_bound(t, layer, s),
                                    f"step {t} layer {layer} seq {s}")
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_q8_draft_step_full_size():
    """q8_0 ring, cap 4096, 5 layers, hidden 4096: prefill then decode steps, sampled heads
    and slots."""
    w = synth.workload(2)
    run = DraftRun(w, 4096, ["full"] * w.n_layer, kv_format="q8_0")
    try:
        heads = [0, 17, 31]
        for t, c in enumerate(synth.commit_schedule(w, 2)):
            outs = run.step(t, c)
            for layer in (0, 4):
                want = run.expected_draft(t, layer, 0, heads=heads)
                assert_close_q8(outs[layer][0][:, heads], want[:, heads],
                                run.draft_bound(t, layer, 0)[:, heads], f"step {t} layer {layer}")
        rng = np.random.default_rng(1)
        run.check_kv(0, 3, list(rng.choice(w.cap, 48, replace=False)))
        assert run.ring.device_error() == 0
    finally:
        run.close()
