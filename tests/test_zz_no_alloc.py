"""ring_attend_static: the allocation-free attention entry point.

Callers that cannot allocate device memory (their framework owns every allocation, or
they run where a runtime allocation is not allowed) get the attention step through an
entry point that takes every buffer from them and keeps its scratch in a fixed static
device array.  Here, on two calls in a row per case, its output must match the existing
entry point's (ring_attend) and the float64 oracle's, within the attention tolerance of
the other GPU tests; the noise rows it writes into the caller's K/V must equal the ones
ring_attend stored, and no other slot may change; and its device error word must read
clear.  This file is collected last, and also passes on its own in a fresh process.
"""

import numpy as np
import pytest
import torch

import synth
from speculative_decoding_draft_kv_gb300 import ring as R
from tests.ring_harness import GpuRun, assert_close

pytestmark = pytest.mark.gpu


def _static_inputs(run, layer, kind):
    """The ring's K/V of one layer (as read back) and its mask of `kind`, in the layouts
    the static entry point takes, on the device."""
    w, g = run.w, run.g
    ks, vs, ms = [], [], []
    for s in range(w.n_seq):
        k, v = run.ring.kv(s, layer)                      # [kv_total][kv_row]
        ks.append(k.reshape(g["kv_total"], w.n_head_kv, w.head_dim).transpose(1, 0, 2))
        vs.append(v.reshape(g["kv_total"], w.n_head_kv, w.head_dim).transpose(1, 0, 2))
        ms.append(run.ring.mask(s, kind))
    dev = run.dev
    k = torch.from_numpy(np.ascontiguousarray(np.stack(ks))).to(dev)
    v = torch.from_numpy(np.ascontiguousarray(np.stack(vs))).to(dev)
    mask = torch.from_numpy(np.stack(ms)).to(dev)
    return k, v, mask


@pytest.mark.parametrize("n_seq,cap,kind,seqs", [
    (1, 4096, "full", [0]),
    (3, 1000, "full", [0, 1, 2]),
    (3, 1000, "swa", [0, 2]),
    # 64 rings: the first split tried needs ~24 MiB of partials, more than the scratch
    # holds, so the call halves its splits until the rest fits (one CTA per kv head)
    (64, 4096, "full", [0, 63]),
])
def test_static_attend_matches_ring_attend_on_two_calls(n_seq, cap, kind, seqs):
    w = synth.workload(2, cap=cap, n_layer=2, n_seq=n_seq, swa_window=min(cap // 2, 2048))
    run = GpuRun(w)
    try:
        assert R.ring_attend_static_device_error() == 0
        sched = synth.commit_schedule(w, 3)
        q_len = w.q_len
        for t, c in enumerate(sched):
            run.begin_step(c)
            if t == 0:
                continue                                   # prefill; then two checked calls
            layer = t % w.n_layer
            q, kn, vn = run.inputs(t, layer, run.dev)
            # the caller's K/V before the call, with the noise slots cleared so that the
            # check below sees what the static call itself writes there
            k, v, mask = _static_inputs(run, layer, kind)
            k[:, :, cap:cap + q_len] = 0
            v[:, :, cap:cap + q_len] = 0
            k_before, v_before = k.clone(), v.clone()
            o_ring = torch.empty_like(q)
            run.ring.attend(layer, kind, q, kn, vn, o_ring)
            torch.cuda.synchronize()
            k_ring, v_ring, _ = _static_inputs(run, layer, kind)
            o_static = torch.full_like(q, float("nan"))
            R.ring_attend_static(w.cap, w.q_len, w.n_head_kv, w.n_head, w.rope_theta,
                                 run.committed, k, v, mask, q, kn, vn, o_static)
            torch.cuda.synchronize()
            assert torch.isfinite(o_static).all()
            got = o_static.cpu().numpy()
            assert_close(got, o_ring.cpu().numpy(), f"call {t} vs ring_attend")
            heads = None if n_seq < 8 else [0, 13, 31]
            for s in seqs:
                want = run.expected(t, layer, kind, s, heads=heads)
                sel = slice(None) if heads is None else heads
                assert_close(got[s][:, sel], want[:, sel], f"call {t} seq {s} vs the oracle")
            # noise slots: exactly ring_attend's rows; every other slot untouched
            noise = slice(cap, cap + q_len)
            assert torch.equal(k[:, :, noise], k_ring[:, :, noise])
            assert torch.equal(v[:, :, noise], v_ring[:, :, noise])
            k_before[:, :, noise] = k_ring[:, :, noise]
            v_before[:, :, noise] = v_ring[:, :, noise]
            assert torch.equal(k, k_before) and torch.equal(v, v_before)
            assert R.ring_attend_static_device_error() == 0
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
    assert R.ring_attend_static_device_error() == 0
