"""GPU parity of ring_step -- the whole step replayed as one CUDA graph -- against the
float64 oracle, with the persistent whole-step attention kernel (few sequences) and with
one attention launch per layer; the layer order it keeps; its bounded waits; the kernel
clock; and long runs (hundreds of steps) whose slot map, masks and tile flags must stay
bit-exact.

Bar: slot_pos, masks and tile flags bit-exact; attention within max-abs 2e-3 and relative
L2 1e-3 of dense float64 attention over exactly the window [lo, committed) plus the noise
block (page "DFLASH2_RING_PORT.md", sections 1.2-1.4 and 1.7).
"""

import time

import numpy as np
import pytest
import torch

import synth
from oracle import ring_oracle as orc
from speculative_decoding_draft_kv_gb300 import ring as R
from tests.ring_harness import GpuRun, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_draft_kv_gb300 import build
    build.build()
    R.library()
    torch.cuda.init()


def _layer_inputs(run, t):
    ins = [run.inputs(t, layer, run.dev) for layer in range(run.w.n_layer)]
    return [x[0] for x in ins], [x[1] for x in ins], [x[2] for x in ins]


def _check_step(run, t, kind, o, seqs=None, heads=None):
    w = run.w
    for layer in range(w.n_layer):
        got = o[layer].cpu().numpy()
        for s in (range(w.n_seq) if seqs is None else seqs):
            want = run.expected(t, layer, kind, s, heads=heads)
            sel = slice(None) if heads is None else heads
            assert_close(got[s][:, sel], want[:, sel], f"step {t} layer {layer} seq {s} {kind}")


def test_step_kernel_steady_decode_full_size():
    """Workload 2 (cap 4096, one sequence, 5 layers): every layer of every step through
    the persistent kernel against the dense float64 window."""
    w = synth.workload(2)
    run = GpuRun(w, step_split=-1)
    try:
        assert run.g["step_split"] > 1 and run.g["step_ctas"] == run.g["step_split"] * w.n_head_kv
        sched = synth.commit_schedule(w, 6)
        assert run.begin_step(sched[0]) == ["bulk"]
        o = [torch.empty((w.n_seq, w.q_len, w.n_head, w.head_dim), device=run.dev)
             for _ in range(w.n_layer)]
        for t in range(1, len(sched)):
            q, kn, vn = _layer_inputs(run, t)
            for x in o:
                x.fill_(float("nan"))
            assert run.step(sched[t], "full", q, kn, vn, o) == ["fold"]
            torch.cuda.synchronize()
            run.check_slots_and_masks()
            _check_step(run, t, "full", o)
        rng = np.random.default_rng(3)
        for layer in (0, 4):
            run.check_kv_slots(0, layer, list(rng.choice(w.cap, 64, replace=False)))
        assert run.ring.device_error() == 0
    finally:
        run.close()


@pytest.mark.parametrize("step_split", [-1, 0])
def test_layers_run_in_order(step_split):
    """Layer l+1's queries are layer l's output buffer (o[l] is q[l+1]), so a layer that
    read its queries before the previous layer had written every output would see the NaNs
    the buffers start with, or a stale step's values.  Each layer is checked against the
    oracle fed with the query it was given: the previous layer's output as read back."""
    w = synth.workload(2, cap=1024, n_layer=4)
    run = GpuRun(w, step_split=step_split)
    try:
        assert (run.g["step_split"] > 0) == (step_split == -1)
        sched = synth.commit_schedule(w, 4)
        run.begin_step(sched[0])
        shape = (w.n_seq, w.q_len, w.n_head, w.head_dim)
        bufs = [torch.empty(shape, device=run.dev) for _ in range(w.n_layer + 1)]
        for t in range(1, len(sched)):
            q0, kn, vn = _layer_inputs(run, t)
            for b in bufs:
                b.fill_(float("nan"))
            bufs[0].copy_(q0[0])
            run.step(sched[t], "full", bufs[:w.n_layer], kn, vn, bufs[1:])
            torch.cuda.synchronize()
            outs = [b.cpu().numpy() for b in bufs]
            for layer in range(w.n_layer):
                assert np.isfinite(outs[layer + 1]).all(), (t, layer)
                want = orc.attend_dense(int(run.committed[0]), w.cap, run.rows.fn(0, layer),
                                        outs[layer][0].astype(np.float64),
                                        kn[layer][0].cpu().numpy(), vn[layer][0].cpu().numpy(),
                                        w.head_dim, w.n_head_kv, w.n_head, w.rope_theta)
                # the query is the float32 output of the layer before, rounded to F16 by the
                # kernel exactly as any query is
                assert_close(outs[layer + 1][0], want, f"step {t} layer {layer}")
        assert run.ring.device_error() == 0
    finally:
        run.close()


@pytest.mark.parametrize("cap,n_seq,step_split,q_len,n_head,swa", [
    (1024, 2, -1, 8, 32, 300),     # chosen split, both masks
    (1024, 2, 1, 8, 32, 300),      # one CTA per pair: every tile in one chunk
    (1024, 1, 5, 8, 32, 0),        # chunks of 3-4 tiles
    (1024, 1, 12, 8, 32, 0),       # the widest cluster: one or two tiles per CTA
    (60, 1, 2, 8, 32, 20),         # noise slots cap..cap+7 straddle two tiles and two CTAs
    (4, 1, 1, 8, 32, 2),           # a ring smaller than one tile
    (1000, 1, -1, 1, 32, 300),      # one query row per head
    (1000, 1, -1, 5, 32, 300),      # ragged row blocks
    (1000, 1, -1, 3, 64, 300),      # eight query heads per kv head
    (1000, 1, -1, 8, 16, 300),      # two query heads per kv head: half the rows
])
def test_step_kernel_splits_and_shapes(cap, n_seq, step_split, q_len, n_head, swa):
    """Any chunking of the tiles over CTAs, any query-row shape, both masks, small rings
    and noise tiles straddling CTAs: outputs within the bar of the oracle, ring state
    bit-exact, and ring_step's state equal to that of the separate calls."""
    w = synth.workload(3, cap=cap, n_layer=3, n_seq=n_seq, q_len=q_len, n_head=n_head,
                       swa_window=swa, extra={"jump_max": 3 * cap, "fold_max": 2 * q_len + 2,
                                              "p_jump": 0.2})
    run = GpuRun(w, step_split=step_split)
    ref = GpuRun(w, step_split=0)
    try:
        assert run.g["step_split"] > 0
        assert ref.g["step_split"] == 0
        kinds = ["full", "swa"] if swa else ["full"]
        shape = (w.n_seq, w.q_len, w.n_head, w.head_dim)
        o = [torch.empty(shape, device=run.dev) for _ in range(w.n_layer)]
        o_ref = [torch.empty(shape, device=run.dev) for _ in range(w.n_layer)]
        for t, c in enumerate(synth.commit_schedule(w, 8)):
            kind = kinds[t % len(kinds)]
            q, kn, vn = _layer_inputs(run, t)
            run.step(c, kind, q, kn, vn, o)
            ref.step(c, kind, q, kn, vn, o_ref)
            torch.cuda.synchronize()
            run.check_slots_and_masks()
            _check_step(run, t, kind, o)
            for layer in range(w.n_layer):
                assert_close(o[layer].cpu().numpy(), o_ref[layer].cpu().numpy(), f"step {t} vs calls")
            for s in range(w.n_seq):
                np.testing.assert_array_equal(run.ring.slot_pos(s), ref.ring.slot_pos(s))
                ka, va = run.ring.kv(s, w.n_layer - 1)
                kb, vb = ref.ring.kv(s, w.n_layer - 1)
                assert np.array_equal(ka.view(np.uint16), kb.view(np.uint16))
                assert np.array_equal(va.view(np.uint16), vb.view(np.uint16))
        assert run.ring.device_error() == 0 and ref.ring.device_error() == 0
    finally:
        run.close()
        ref.close()


def test_step_split_requests_that_cannot_run_are_refused():
    w = synth.workload(2, cap=1024, n_layer=2)
    with pytest.raises(R.RingError) as e:            # more CTAs than fit on the GPU at once
        R.Ring(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer, w.rope_theta,
               step_split=1000)
    assert e.value.code == R.RING_EINVAL
    with pytest.raises(R.RingError) as e:            # q8_0 slots take one launch per layer
        R.Ring(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer, w.rope_theta,
               step_split=2, kv_format="q8_0")
    assert e.value.code == R.RING_EINVAL
    with R.Ring(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, 17, w.rope_theta,
                step_split=-1) as r:
        assert r.geometry["step_split"] == 0         # more layers than one launch takes


@pytest.mark.parametrize("which,bit", [(0, 1), (1, 16)])
def test_bounded_waits_run_out_and_return(which, bit):
    """A wait on an mbarrier nobody arrives at (0), or on a counter no CTA raises (1),
    gives up after its limit, sets its bit in the device error word and lets the kernel
    return; the context stays usable."""
    w = synth.workload(1, cap=64, n_layer=1)
    run = GpuRun(w)
    try:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        run.ring.check_bounded_wait(which, 2000)          # 2 ms
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        assert 0.002 <= dt < 1.0, dt
        assert run.ring.device_error() == bit
        assert run.ring.device_error() == 0              # read and cleared
        run.begin_step([30])
        got = run.attend(0, 0, "full")
        assert_close(got[0], run.expected(0, 0, "full", 0), "after the probe")
        with pytest.raises(R.RingError) as e:
            run.ring.check_bounded_wait(2, 10)
        assert e.value.code == R.RING_EINVAL
        with pytest.raises(R.RingError) as e:
            run.ring.check_bounded_wait(0, 0)
        assert e.value.code == R.RING_EINVAL
    finally:
        run.close()


@pytest.mark.parametrize("step_split", [-1, 0])
def test_kernel_clock_counts_launches(step_split):
    """The device-side clock of the attention kernel records one launch per step (the
    persistent kernel) or one per layer, and its time fits inside the step's event time."""
    w = synth.workload(2, cap=1024, n_layer=3)
    run = GpuRun(w, step_split=step_split)
    try:
        sched = synth.commit_schedule(w, 12)
        run.begin_step(sched[0])
        shape = (w.n_seq, w.q_len, w.n_head, w.head_dim)
        o = [torch.empty(shape, device=run.dev) for _ in range(w.n_layer)]
        q, kn, vn = _layer_inputs(run, 1)
        run.ring.clock_enable(True)
        assert run.ring.clock_read() == (0.0, 0)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for t in range(1, len(sched)):
            run.step(sched[t], "full", q, kn, vn, o)
        b.record()
        torch.cuda.synchronize()
        ms, n = run.ring.clock_read()
        per_step = 1 if step_split == -1 else w.n_layer
        assert n == per_step * (len(sched) - 1)
        assert 0.0 < ms <= a.elapsed_time(b)
        run.ring.clock_enable(False)
        run.step(sched[-1], "full", q, kn, vn, o)
        assert run.ring.clock_read() == (0.0, 0)
        assert run.ring.device_error() == 0
    finally:
        run.close()


@pytest.mark.parametrize("wid,n_steps,seqs,step_split", [(2, 500, None, 0), (2, 300, None, -1),
                                                         (5, 200, [0, 6, 15], 0)])
def test_long_run_state_stays_bit_exact(wid, n_steps, seqs, step_split):
    """Hundreds of ring_step calls (slots overwritten round-robin, section 1.2): slot_pos,
    both masks and the tile flags bit for bit against the bookkeeping oracle at
    checkpoints, and every layer's attention on the last step against the oracle."""
    w = synth.workload(wid)
    run = GpuRun(w, swa_window=2048, step_split=step_split)
    try:
        sched = synth.commit_schedule(w, n_steps)
        run.begin_step(sched[0])
        q, kn, vn = _layer_inputs(run, 0)
        o = [torch.empty((w.n_seq, w.q_len, w.n_head, w.head_dim), device=run.dev)
             for _ in range(w.n_layer)]
        checkpoints = {1, n_steps // 3, 2 * n_steps // 3}
        for t in range(1, n_steps):
            last = t == n_steps - 1
            if last:
                q, kn, vn = _layer_inputs(run, t)
            run.step(sched[t], "full", q, kn, vn, o)
            if t in checkpoints or last:
                run.check_slots_and_masks(seqs=seqs)
        torch.cuda.synchronize()
        assert run.committed.min() >= w.cap          # the ring has wrapped
        heads = None if seqs is None else [0, 17, 31]
        _check_step(run, n_steps - 1, "full", o, seqs=[0] if seqs is None else seqs[:2], heads=heads)
        assert run.ring.device_error() == 0
    finally:
        run.close()
