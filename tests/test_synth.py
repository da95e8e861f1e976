"""The seeded input generator and the workload schedules (CPU)."""

import numpy as np
import torch

import synth


def test_values_are_deterministic_and_roughly_normal():
    keys = torch.arange(4000, dtype=torch.int64) * 7919
    a = synth.gaussian_values(keys, 256, 0.5)
    b = synth.gaussian_values(keys, 256, 0.5)
    assert torch.equal(a, b)
    x = a.double()
    assert abs(x.mean().item()) < 0.005
    assert abs(x.std().item() - 0.5) < 0.005
    assert x.abs().max().item() <= 0.5 * 3.4642
    # roughly Gaussian tails: about 4.55 % beyond 2 sigma (Irwin-Hall(4) gives ~4.2 %)
    frac = (x.abs() > 1.0).double().mean().item()
    assert 0.035 < frac < 0.05


def test_streams_and_positions_are_distinct():
    w = synth.workload(2)
    k, v = synth.context_rows(w.seed, 0, 0, torch.arange(64), w.kv_row, w.sigma)
    assert k.dtype == torch.float16 and k.shape == (64, 1024)
    assert not torch.equal(k, v)
    assert len({tuple(r[:8].tolist()) for r in k}) == 64
    k2, _ = synth.context_rows(w.seed, 1, 0, torch.arange(64), w.kv_row, w.sigma)
    assert not torch.equal(k, k2)
    q = synth.query_block(w.seed, 3, 0, 1, 8, 32, 128, 0.5)
    assert q.shape == (8, 32, 128) and q.dtype == torch.float32
    kn, vn = synth.noise_rows(w.seed, 3, 0, 1, 8, 1024, 0.5)
    assert kn.shape == (8, 1024) and not torch.equal(kn, vn)


def test_hash32_matches_plain_integer_arithmetic():
    def ref(x):
        x &= 0xFFFFFFFF
        x ^= x >> 16
        x = (x * 0x7FEB352D) & 0xFFFFFFFF
        x ^= x >> 15
        x = (x * 0x846CA68B) & 0xFFFFFFFF
        x ^= x >> 16
        return x
    xs = [0, 1, 2, 0xFFFFFFFF, 0x12345678, 0x80000000, 0xDEADBEEF]
    got = synth.hash32(torch.tensor(xs, dtype=torch.int64)).tolist()
    assert got == [ref(x) for x in xs]
    assert [synth.hash32(x) for x in xs] == [ref(x) for x in xs]


def test_schedules_follow_their_workload():
    s1 = synth.commit_schedule(synth.workload(1))
    inc = np.diff(np.concatenate([[0], s1[:, 0]]))
    assert s1.shape == (40, 1) and inc.min() >= 1 and inc.max() <= 9
    assert 120 < s1[-1, 0] < 280                       # grows to ~200: wraps cap 64 a few times
    s2 = synth.commit_schedule(synth.workload(2), 20000)
    assert s2[0, 0] == 8192
    inc = np.diff(s2[:, 0])
    hist = np.bincount(inc - 1, minlength=8) / len(inc)
    want = np.array([24.5, 19.5, 15.0, 9.9, 7.7, 5.0, 3.6, 14.7])
    np.testing.assert_allclose(hist, want / want.sum(), atol=0.01)
    s3 = synth.commit_schedule(synth.workload(3))
    d3 = np.diff(s3[:, 0])
    assert (d3 > 18).any() and (d3 <= 18).any() and d3.max() <= 30000
    s4 = synth.commit_schedule(synth.workload(4), 10)
    assert s4.shape == (11, 64) and s4[0].min() >= 1 and s4[0].max() <= 131072
    s5 = synth.commit_schedule(synth.workload(5), 10)
    assert s5.shape == (11, 16) and s5[0].min() >= 131072


def test_feature_rows_and_producer_weights_are_pure_functions():
    a = synth.feature_rows(7, 1, torch.arange(10, 20), 256, 0.5)
    b = synth.feature_rows(7, 1, torch.tensor([15, 12]), 256, 0.5)
    assert torch.equal(a[5], b[0]) and torch.equal(a[2], b[1])
    assert not torch.equal(a[0], synth.feature_rows(7, 2, torch.tensor([10]), 256, 0.5)[0])
    wk, wv, kn = synth.producer_weights(7, 3, 64, 256, 16)
    wk2, wv2, kn2 = synth.producer_weights(7, 3, 64, 256, 16)
    assert torch.equal(wk, wk2) and torch.equal(wv, wv2) and torch.equal(kn, kn2)
    assert wk.dtype == torch.float16 and kn.dtype == torch.float32 and kn.shape == (16,)
    assert not torch.equal(wk, wv)
    assert abs(float(wk.float().std()) - 1 / 16) < 0.01
    assert not torch.equal(wk, synth.producer_weights(7, 4, 64, 256, 16)[0])
