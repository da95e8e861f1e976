"""GPU parity of the q8_0 ring (through the C ABI) against the float64 oracle.

Slots hold q8_0 blocks (32 values: int8 codes and one F16 scale).  Bar: slot_pos, masks
and tile flags bit-exact; V codes and scales bit-exact (both sides take the float32
decisions on the same F16 inputs); K codes within one and K scales within one F16 ulp,
on at most 1 % of the codes (the GPU rotates in float32, the oracle in float64); pad rows
all-zero blocks; attention within max-abs 2e-3 and relative L2 1e-3 of dense float64
attention over the dequantised window plus the dequantised noise block.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import ring_oracle as orc
from speculative_decoding_draft_kv_gb300 import ring as R
from tests.ring_harness import GpuRun, assert_close, q8_k_within

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_draft_kv_gb300 import build
    build.build()
    R.library()
    torch.cuda.init()


def _state_matches(run, full, layers):
    """Whole q8_0 ring state of sequence 0 against the step-by-step oracle."""
    n_diff = n_all = 0
    for layer in layers:
        kc, ks, vc, vs = run.ring.kv_q8(0, layer)
        np.testing.assert_array_equal(vc, full.vq[layer])
        np.testing.assert_array_equal(vs.view(np.uint16), full.vs[layer].view(np.uint16))
        n_diff += q8_k_within(kc, ks, full.kq[layer], full.ks[layer])
        n_all += kc.size
    return n_diff, n_all


@pytest.mark.parametrize("tps", [0, 1])
def test_q8_tiny_ring_full_state_parity(tps):
    """Workload 1 (cap 64, 1 layer, 40 steps) on a q8_0 ring: the whole ring state (codes
    and scales of every slot, noise slots and trash slot included) after every step and
    every attention output, both masks."""
    w = synth.workload(1, swa_window=24)
    run = GpuRun(w, tiles_per_split=tps, kv_format="q8_0")
    full = orc.RingOracle(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer,
                          w.rope_theta, swa_window=w.swa_window, kv_format="q8_0")
    n_diff = n_all = 0
    try:
        assert " q8_0 cache " in run.ring.describe()
        for t, c in enumerate(synth.commit_schedule(w)):
            run.begin_step(c)
            st, _ = full.rows_needed(int(c[0]))
            k, v = run.rows.rows(0, 0, np.arange(st, int(c[0])))
            full.begin_step(int(c[0]), k[None], v[None], st)
            run.check_slots_and_masks()
            for kind in ("full", "swa"):
                o = run.attend(t, 0, kind)
                q, kn, vn = [x[0].cpu().numpy() for x in run.inputs(t, 0, "cpu")]
                o1 = full.attend(0, q, kn, vn, kind)
                o2 = run.expected(t, 0, kind, 0)
                assert np.abs(o1 - o2).max() < 1e-12
                assert_close(o[0], o2, f"step {t} {kind}")
            a, b = _state_matches(run, full, [0])
            n_diff += a
            n_all += b
        assert n_diff <= 0.01 * n_all
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_q8_steady_decode_parity_full_size():
    """Workload 2 at full size (cap 4096, 5 layers) on a q8_0 ring: prefill through the
    bulk path, then decode steps; every layer's output and sampled slots checked."""
    w = synth.workload(2)
    run = GpuRun(w, kv_format="q8_0")
    try:
        g = run.g
        assert g["cluster"] > 1          # one sequence: the cluster shape
        assert g["cache_bytes"] == 2 * w.n_layer * g["kv_total"] * (w.kv_row + w.kv_row // 32 * 2)
        sched = synth.commit_schedule(w, 6)
        assert run.begin_step(sched[0]) == ["bulk"]
        run.check_slots_and_masks()
        for t in range(1, len(sched)):
            assert run.begin_step(sched[t]) == ["fold"]
            run.check_slots_and_masks()
            for layer in range(w.n_layer):
                o = run.attend(t, layer, "full")
                assert_close(o[0], run.expected(t, layer, "full", 0), f"step {t} layer {layer}")
        rng = np.random.default_rng(0)
        for layer in (0, 4):
            run.check_kv_slots_q8(0, layer, list(rng.choice(w.cap, 64, replace=False)))
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_q8_batched_rings_parity_full_size():
    """Workload 4 (64 rings, ragged committed counts, SWA window 2048) on q8_0 rings:
    both masks, outputs sampled per sequence, slots sampled."""
    w = synth.workload(4)
    run = GpuRun(w, kv_format="q8_0")
    try:
        sched = synth.commit_schedule(w, 2)
        for t in range(len(sched)):
            run.begin_step(sched[t])
            run.check_slots_and_masks(seqs=[0, 17, 63])
        t = len(sched) - 1
        for kind in ("full", "swa"):
            for layer in (1, 3):
                o = run.attend(t, layer, kind)
                for s in (0, 17, 63):
                    heads = [0, 5, 31]
                    want = run.expected(t, layer, kind, s, heads=heads)
                    assert_close(o[s][:, heads], want[:, heads], f"seq {s} {kind} layer {layer}")
        run.check_kv_slots_q8(5, 2, list(range(0, w.cap, 97)))
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_q8_large_ring_parity_full_size():
    """Workload 5 (16 rings of cap 32768, wrapped four times) on q8_0 rings."""
    w = synth.workload(5)
    run = GpuRun(w, kv_format="q8_0")
    try:
        sched = synth.commit_schedule(w, 2)
        for t in range(len(sched)):
            run.begin_step(sched[t])
            run.check_slots_and_masks(seqs=[0, 7, 15])
        t = len(sched) - 1
        o = run.attend(t, 2, "full")
        for s in (0, 15):
            heads = [3, 30]
            want = run.expected(t, 2, "full", s, heads=heads)
            assert_close(o[s][:, heads], want[:, heads], f"seq {s}")
        run.check_kv_slots_q8(15, 2, list(range(0, w.cap, 511)))
        assert run.ring.device_error() == 0
    finally:
        run.close()


@pytest.mark.parametrize("cap,tps", [(60, 1), (60, 0), (4, 0), (200, 1), (1000, 2)])
def test_q8_noise_tiles_and_small_rings(cap, tps):
    """q8_0 slots where the noise block straddles two tiles owned by two CTAs (cap 60), a
    ring smaller than one tile (cap 4) and a ragged last tile of 32 slots."""
    w = synth.workload(1, cap=cap, n_layer=2, swa_window=max(2, cap // 3))
    run = GpuRun(w, tiles_per_split=tps, kv_format="q8_0")
    try:
        for t, c in enumerate(synth.commit_schedule(w, 12)):
            run.begin_step(c)
            run.check_slots_and_masks()
            for kind in ("full", "swa"):
                layer = t % 2
                o = run.attend(t, layer, kind)
                assert_close(o[0], run.expected(t, layer, kind, 0), f"cap {cap} step {t} {kind}")
        run.check_kv_slots_q8(0, 1, list(range(cap)))
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_q8_step_graph_matches_separate_calls():
    """ring_step (one replayed CUDA graph per step) on q8_0 rings gives the same outputs
    and the same codes and scales as ring_begin_step + ring_attend per layer, through
    fold-in steps, bulk steps and both masks."""
    w = synth.workload(3, cap=512, n_layer=3, n_seq=2, swa_window=100,
                       extra={"jump_max": 3000, "fold_max": 18, "p_jump": 0.3})
    a, b = GpuRun(w, kv_format="q8_0"), GpuRun(w, kv_format="q8_0")
    try:
        L = w.n_layer
        outs = [[torch.empty((w.n_seq, w.q_len, w.n_head, w.head_dim), device=a.dev) for _ in range(L)]
                for _ in range(2)]
        for t, c in enumerate(synth.commit_schedule(w, 8)):
            kind = "swa" if t % 3 == 2 else "full"
            a.begin_step(c)
            k_rows, v_rows = a._keep
            row_off, first = [], []
            n = 0
            for s in range(w.n_seq):
                st, nn = b.ring.rows_needed(s, int(c[s]))
                row_off.append(n)
                first.append(st)
                n += nn
            ins = [a.inputs(t, layer, a.dev) for layer in range(L)]
            o_ref = []
            for layer in range(L):
                o = torch.empty_like(ins[layer][0])
                a.ring.attend(layer, kind, *ins[layer], o)
                o_ref.append(o)
            o_graph = outs[t % 2]
            b.ring.step(c, k_rows, v_rows, row_off, first, kind, [x[0] for x in ins],
                        [x[1] for x in ins], [x[2] for x in ins], o_graph)
            torch.cuda.synchronize()
            for layer in range(L):
                assert torch.equal(o_graph[layer], o_ref[layer]), (t, layer)
            for s in range(w.n_seq):
                for x, y in zip(a.ring.kv_q8(s, L - 1), b.ring.kv_q8(s, L - 1)):
                    assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
        assert a.ring.device_error() == 0 and b.ring.device_error() == 0
    finally:
        a.close()
        b.close()


def test_q8_host_errors():
    """Calls that a q8_0 ring refuses, and an unknown format."""
    w = synth.workload(1)
    with pytest.raises(R.RingError):
        R.Ring(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer, w.rope_theta,
               kv_format=7)
    with R.Ring(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer, w.rope_theta,
                kv_format="q8_0") as r:
        with pytest.raises(R.RingError):
            r.kv(0, 0)
        kc, ks, vc, vs = r.kv_q8(0, 0)
        assert not kc.any() and not vc.any()
    with R.Ring(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer, w.rope_theta) as r:
        with pytest.raises(R.RingError):
            r.kv_q8(0, 0)
