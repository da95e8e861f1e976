"""GPU parity of the CUDA ring step (through the C ABI) against the float64 oracle.

Bar: slot_pos, masks and tile flags bit-exact; V slots and the trash slot bit-exact;
K slots within one binary16 ulp (the GPU rounds the same float64 rotation, with CUDA's
own sin/cos); attention within max-abs 2e-3 and relative L2 1e-3 of dense float64
attention over exactly the window [lo, committed) plus the noise block.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import ring_oracle as orc
from speculative_decoding_draft_kv_gb300 import ring as R
from tests.ring_harness import GpuRun, assert_close, k_within_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_draft_kv_gb300 import build
    build.build()
    R.library()
    torch.cuda.init()


def test_generator_is_bit_identical_on_cpu_and_gpu():
    w = synth.workload(5)
    pos = torch.tensor([0, 1, 777, 131071, 140000])
    kc, vc = synth.context_rows(w.seed, 3, 4, pos, w.kv_row, w.sigma)
    kg, vg = synth.context_rows(w.seed, 3, 4, pos.cuda(), w.kv_row, w.sigma, device="cuda")
    assert torch.equal(kc, kg.cpu()) and torch.equal(vc, vg.cpu())
    qc = synth.query_block(w.seed, 9, 2, 1, 8, 32, 128, w.sigma)
    qg = synth.query_block(w.seed, 9, 2, 1, 8, 32, 128, w.sigma, device="cuda")
    assert torch.equal(qc, qg.cpu())


def test_geometry_and_describe_line():
    w = synth.workload(2)
    with R.Ring(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer, w.rope_theta) as r:
        g = r.geometry
        assert (g["a_step"], g["trash_slot"], g["kv_total"], g["kv_row"]) == (18, 4104, 4128, 1024)
        assert g["cache_bytes"] == 84_541_440
        assert r.describe().endswith("cap=4096 kv_total=4128 a_step=18 layers=5 f16 cache 80.6 MiB")
        assert (r.slot_pos() == -1).all()


def test_tiny_ring_full_state_parity():
    """Workload 1 (cap 64, 1 layer, 40 steps): the whole ring state after every step and
    every attention output, both masks, against the step-by-step oracle and the dense
    window oracle."""
    w = synth.workload(1, swa_window=24)
    run = GpuRun(w)
    full = orc.RingOracle(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer,
                          w.rope_theta, swa_window=w.swa_window)
    k_not_exact = k_total = 0
    try:
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
            gk, gv = run.ring.kv(0, 0)
            np.testing.assert_array_equal(gv, full.v[0])
            ok, inexact = k_within_tolerance(gk, full.k[0])
            assert ok
            k_not_exact += inexact
            k_total += gk.size
        # the GPU rotates in float32: rarely it lands on the other side of an F16 rounding
        assert k_not_exact <= 0.01 * k_total
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_steady_decode_parity_full_size():
    """Workload 2 at full size: prefill 8192 through the bulk path, then decode steps
    drawn from the acceptance histogram; every layer's output checked."""
    w = synth.workload(2)
    run = GpuRun(w)
    try:
        sched = synth.commit_schedule(w, 8)
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
            run.check_kv_slots(0, layer, list(rng.choice(w.cap, 64, replace=False)))
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_bulk_stress_parity_full_size():
    """Workload 3: long jumps (bulk path, ring overwrite) mixed with fold-ins."""
    w = synth.workload(3)
    run = GpuRun(w)
    try:
        paths = []
        rng = np.random.default_rng(1)
        for t, c in enumerate(synth.commit_schedule(w, 10)):
            paths += run.begin_step(c)
            run.check_slots_and_masks()
            layer = t % w.n_layer
            o = run.attend(t, layer, "full")
            assert_close(o[0], run.expected(t, layer, "full", 0), f"step {t}")
            run.check_kv_slots(0, layer, list(rng.choice(w.cap, 32, replace=False)))
        assert "bulk" in paths and "fold" in paths
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_batched_rings_parity_full_size():
    """Workload 4: 64 independent rings with ragged committed counts; mask_full and
    mask_swa (window 2048) both checked; outputs sampled per sequence."""
    w = synth.workload(4)
    run = GpuRun(w)
    try:
        sched = synth.commit_schedule(w, 2)
        for t in range(len(sched)):
            run.begin_step(sched[t])
            run.check_slots_and_masks()
        t = len(sched) - 1
        for kind in ("full", "swa"):
            for layer in (1, 3):
                o = run.attend(t, layer, kind)
                for s in (0, 17, 63):
                    heads = [0, 5, 31]
                    want = run.expected(t, layer, kind, s, heads=heads)
                    assert_close(o[s][:, heads], want[:, heads], f"seq {s} {kind} layer {layer}")
        run.check_kv_slots(5, 2, list(range(0, w.cap, 97)))
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_large_ring_parity_full_size():
    """Workload 5: 16 rings of cap 32768, committed near 131072 (wrapped four times)."""
    w = synth.workload(5)
    run = GpuRun(w)
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
        run.check_kv_slots(15, 2, list(range(0, w.cap, 511)))
        assert run.ring.device_error() == 0
    finally:
        run.close()


@pytest.mark.parametrize("tps,max_cluster", [(0, 0), (0, 1), (0, 2), (1, 0), (3, 0), (3, 1),
                                             (100, 0), (2, 16)])
def test_split_sizes_agree(tps, max_cluster):
    """Any split of the slot tiles -- one CTA, clusters merging through distributed shared
    memory, independent CTAs with a combine kernel, or both -- changes only rounding."""
    w = synth.workload(2, cap=1024, n_layer=2)
    run = GpuRun(w, tiles_per_split=tps, max_cluster=max_cluster)
    try:
        g = run.g
        assert g["n_splits"] == g["cluster"] * g["groups"]
        assert g["n_splits"] * g["tiles_per_split"] >= g["n_tiles"]
        for t, c in enumerate(synth.commit_schedule(w, 3)):
            run.begin_step(c)
            if t >= 2:      # repeated launches reuse the partial buffers
                for layer in (1, 0, 1):
                    o = run.attend(t, layer, "full")
                    assert_close(o[0], run.expected(t, layer, "full", 0),
                                 f"tps {tps} cluster {g['cluster']} groups {g['groups']}")
        assert run.ring.device_error() == 0
    finally:
        run.close()


@pytest.mark.parametrize("q_len,n_head,max_cluster", [(1, 32, 0), (4, 32, 0), (5, 32, 0),
                                                      (7, 32, 0), (8, 16, 0), (3, 64, 0),
                                                      (5, 32, 1)])
def test_query_row_shapes(q_len, n_head, max_cluster):
    """Query blocks of G * q_len rows that fill one or both 16-row blocks of a CTA, or only
    part of them, in clusters and in plain CTAs; SWA included."""
    w = synth.workload(2, cap=1024, n_layer=2, q_len=q_len, n_head=n_head, swa_window=300)
    run = GpuRun(w, max_cluster=max_cluster)
    try:
        for t, c in enumerate(synth.commit_schedule(w, 3)):
            run.begin_step(c)
        run.check_slots_and_masks()
        for kind in ("full", "swa"):
            o = run.attend(3, 1, kind)
            assert_close(o[0], run.expected(3, 1, kind, 0), f"q_len {q_len} heads {n_head} {kind}")
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_bulk_chunk_and_prefill_route_leave_identical_state():
    w = synth.workload(2, cap=512, n_layer=2)
    runs = [GpuRun(w, bulk_chunk=1024), GpuRun(w, bulk_chunk=37), GpuRun(w, bulk_chunk=64)]
    try:
        runs[0].begin_step([1000])
        runs[1].begin_step([1000])
        for c in (100, 300, 512, 700, 1000):        # the same window reached in steps
            runs[2].begin_step([c])
        ref_k, ref_v = runs[0].ring.kv(0, 1)
        for r in runs[1:]:
            np.testing.assert_array_equal(r.ring.slot_pos(), runs[0].ring.slot_pos())
            k, v = r.ring.kv(0, 1)
            np.testing.assert_array_equal(k[:w.cap].view(np.uint16), ref_k[:w.cap].view(np.uint16))
            np.testing.assert_array_equal(v[:w.cap].view(np.uint16), ref_v[:w.cap].view(np.uint16))
    finally:
        for r in runs:
            r.close()


def test_edge_cases_and_host_errors():
    w = synth.workload(1, cap=64, n_layer=2, swa_window=8)
    run = GpuRun(w)
    try:
        q, kn, vn = run.inputs(0, 0, run.dev)
        o = torch.empty_like(q)
        with pytest.raises(R.RingError) as e:            # attend before any begin_step
            run.ring.attend(0, "full", q, kn, vn, o)
        assert e.value.code == R.RING_ESTATE
        assert run.begin_step([0]) == ["fold"]           # empty context: only the noise
        run.check_slots_and_masks()
        for kind in ("full", "swa"):
            got = run.attend(0, 1, kind)
            assert_close(got[0], run.expected(0, 1, kind, 0), kind)
        assert run.begin_step([18]) == ["fold"]          # n_new == a_step: fold-in
        assert run.begin_step([37]) == ["bulk"]          # n_new == a_step + 1: bulk
        assert run.begin_step([37]) == ["fold"]          # nothing new
        run.check_slots_and_masks()
        assert run.begin_step([500]) == ["bulk"]         # jump past the whole ring
        run.check_slots_and_masks()
        got = run.attend(5, 0, "swa")
        assert_close(got[0], run.expected(5, 0, "swa", 0), "after jump")
        before = run.ring.slot_pos().copy()
        with pytest.raises(R.RingError) as e:            # committed went backwards
            run.ring.begin_step([499], None, None, [0], [0])
        assert e.value.code == R.RING_ERANGE
        k = torch.zeros((2, 4, 1024), dtype=torch.float16, device=run.dev)
        with pytest.raises(R.RingError) as e:            # rows do not cover [start, c)
            run.ring.begin_step([510], k, k, [0], [506])
        assert e.value.code == R.RING_ERANGE
        with pytest.raises(R.RingError) as e:            # rows run past n_rows
            run.ring.begin_step([510], k, k, [0], [500])
        assert e.value.code == R.RING_ERANGE
        np.testing.assert_array_equal(run.ring.slot_pos(), before)
        with pytest.raises(R.RingError) as e:
            run.ring.attend(2, "full", q, kn, vn, o)      # layer out of range
        assert e.value.code == R.RING_EINVAL
        assert run.ring.device_error() == 0
    finally:
        run.close()
    nos = GpuRun(synth.workload(1))
    try:
        nos.begin_step([10])
        q, kn, vn = nos.inputs(0, 0, nos.dev)
        with pytest.raises(R.RingError) as e:             # SWA without a window
            nos.ring.attend(0, "swa", q, kn, vn, torch.empty_like(q))
        assert e.value.code == R.RING_EINVAL
    finally:
        nos.close()


@pytest.mark.parametrize("cap,tps", [(60, 1), (60, 0), (4, 0), (200, 1), (1000, 2)])
def test_noise_tiles_and_small_rings(cap, tps):
    """Noise slots cap..cap+7 straddling two tiles owned by two CTAs (cap 60, one tile per
    CTA), a ring smaller than one tile (cap 4), and group-combine splits."""
    w = synth.workload(1, cap=cap, n_layer=2, swa_window=max(2, cap // 3))
    run = GpuRun(w, tiles_per_split=tps)
    try:
        for t, c in enumerate(synth.commit_schedule(w, 12)):
            run.begin_step(c)
            run.check_slots_and_masks()
            for kind in ("full", "swa"):
                layer = t % 2
                o = run.attend(t, layer, kind)
                assert_close(o[0], run.expected(t, layer, kind, 0), f"cap {cap} step {t} {kind}")
        assert run.ring.device_error() == 0
    finally:
        run.close()


def test_step_graph_matches_separate_calls():
    """ring_step with one attention launch per layer (one replayed CUDA graph per step)
    gives the same outputs and the same ring state as ring_begin_step + ring_attend per
    layer, bit for bit, through fold-in steps, a bulk step, a change of the layer buffers
    (re-capture) and both masks.  (The persistent whole-step kernel splits the slots
    differently; tests/test_gpu_step.py holds it to the oracle and to these calls.)"""
    w = synth.workload(3, cap=512, n_layer=3, n_seq=2, swa_window=100,
                       extra={"jump_max": 3000, "fold_max": 18, "p_jump": 0.3})
    a, b = GpuRun(w), GpuRun(w, step_split=0)
    try:
        L = w.n_layer
        outs = [[torch.empty((w.n_seq, w.q_len, w.n_head, w.head_dim), device=a.dev) for _ in range(L)]
                for _ in range(2)]
        for t, c in enumerate(synth.commit_schedule(w, 8)):
            kind = "swa" if t % 3 == 2 else "full"
            # rows for both rings (same values); b takes them through ring_step
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
            o_graph = outs[t % 2]                       # alternate buffers: forces re-capture
            b.ring.step(c, k_rows, v_rows, row_off, first, kind, [x[0] for x in ins],
                        [x[1] for x in ins], [x[2] for x in ins], o_graph)
            z = [np.zeros((1, int(c[s]) - first[s], 2), np.float16) for s in range(w.n_seq)]
            for s in range(w.n_seq):
                b.book[s].begin_step(int(c[s]), z[s], z[s], first[s])
            torch.cuda.synchronize()
            for layer in range(L):
                assert torch.equal(o_graph[layer], o_ref[layer]), (t, layer)
            b.check_slots_and_masks()
            for s in range(w.n_seq):
                ka, va = a.ring.kv(s, L - 1)
                kb, vb = b.ring.kv(s, L - 1)
                assert np.array_equal(ka.view(np.uint16), kb.view(np.uint16))
                assert np.array_equal(va.view(np.uint16), vb.view(np.uint16))
        assert a.ring.device_error() == 0 and b.ring.device_error() == 0
    finally:
        a.close()
        b.close()
