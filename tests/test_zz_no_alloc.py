"""ring_attend_static: the allocation-free attention entry point, against ring_attend.

Callers that cannot allocate device memory (their framework owns every allocation, or
they run where a runtime allocation is not allowed) get the attention step through an
entry point that takes every buffer from them and keeps its scratch in a fixed static
device array.  Here its output must match the existing entry point's output, within the
attention tolerance of the other GPU tests, on two calls in a row -- and the noise rows
it writes into the caller's K/V must equal the ones ring_attend stored.  This file is
collected last, and also passes on its own in a fresh process.
"""

import numpy as np
import pytest
import torch

import synth
from speculative_decoding_draft_kv_gb300 import ring as R
from tests.ring_harness import GpuRun, assert_close

pytestmark = pytest.mark.gpu


def _static_inputs(run, layer):
    """The ring's K/V of one layer (as read back) and its full mask, in the layouts the
    static entry point takes, on the device."""
    w, g = run.w, run.g
    ks, vs, ms = [], [], []
    for s in range(w.n_seq):
        k, v = run.ring.kv(s, layer)                      # [kv_total][kv_row]
        ks.append(k.reshape(g["kv_total"], w.n_head_kv, w.head_dim).transpose(1, 0, 2))
        vs.append(v.reshape(g["kv_total"], w.n_head_kv, w.head_dim).transpose(1, 0, 2))
        ms.append(run.ring.mask(s, "full"))
    dev = run.dev
    k = torch.from_numpy(np.ascontiguousarray(np.stack(ks))).to(dev)
    v = torch.from_numpy(np.ascontiguousarray(np.stack(vs))).to(dev)
    mask = torch.from_numpy(np.stack(ms)).to(dev)
    return k, v, mask


@pytest.mark.parametrize("n_seq,cap", [(1, 4096), (3, 1000)])
def test_static_attend_matches_ring_attend_on_two_calls(n_seq, cap):
    w = synth.workload(2, cap=cap, n_layer=2, n_seq=n_seq)
    run = GpuRun(w)
    try:
        sched = synth.commit_schedule(w, 3)
        for t, c in enumerate(sched):
            run.begin_step(c)
            if t == 0:
                continue                                   # prefill; then two checked calls
            layer = t % w.n_layer
            q, kn, vn = run.inputs(t, layer, run.dev)
            o_ring = torch.empty_like(q)
            run.ring.attend(layer, "full", q, kn, vn, o_ring)
            torch.cuda.synchronize()
            k, v, mask = _static_inputs(run, layer)
            k_before, v_before = k.clone(), v.clone()
            o_static = torch.full_like(q, float("nan"))
            R.ring_attend_static(w.cap, w.q_len, w.n_head_kv, w.n_head, w.rope_theta,
                                 run.committed, k, v, mask, q, kn, vn, o_static)
            torch.cuda.synchronize()
            assert torch.isfinite(o_static).all()
            assert_close(o_static.cpu().numpy(), o_ring.cpu().numpy(), f"call {t}")
            # the noise rows it wrote equal those ring_attend stored (the rest untouched)
            assert torch.equal(k, k_before) and torch.equal(v, v_before)
    finally:
        run.close()


def test_static_attend_rejects_bad_shapes():
    dev = torch.device("cuda")
    q = torch.zeros((1, 8, 32, 128), device=dev)
    kv = torch.zeros((1, 8, 96, 128), dtype=torch.float16, device=dev)
    mask = torch.zeros((1, 8, 96), device=dev)
    noise = torch.zeros((1, 8, 1024), dtype=torch.float16, device=dev)
    with pytest.raises(R.RingError) as e:                 # head group * q_len above 32 rows
        R.ring_attend_static(64, 8, 4, 32, 1e6, [10], kv, kv, mask, q, noise, noise, q.clone())
    assert e.value.code == R.RING_EINVAL
    big = torch.zeros((300, 1, 1, 1), device=dev)
    with pytest.raises(R.RingError) as e:                 # more sequences than supported
        R.ring_attend_static(64, 8, 8, 32, 1e6, [1] * 300, kv, kv, mask, big, noise, noise, big)
    assert e.value.code == R.RING_ERANGE
