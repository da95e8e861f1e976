"""GPU parity when the attention scores span a range far wider than the exponent of one
float32 or F16 value, through the C ABI against the float64 oracle.

The online softmax of a split-KV decode kernel keeps a reference maximum per query row;
the kernels move it lazily (only when a row outgrows it by more than 2^8), so the
probabilities they round to F16 range over [0, 256].  Ordinary synthetic rows move the
reference almost only on a row's first tile.  Here the keys carry a staircase along the
last rotary pair (dimensions 63 and 127 of each head, which RoPE turns by at most a few
milliradians over the window): k[63] = 127 j / 16 on level j = -16 .. 16 of cap / 32
positions each, the queries +-7.375 in dimension 63.  One level raises a score by 7.46
log2 units, so a row's reference stays put over one level (P up to ~2^7.5) and moves on the
next; the scores span ~166 natural units, beyond float32's exponent range.  Query heads
of alternating sign put the maximum at the newest or at the oldest positions, so inside
one warp some rows move their reference and others never do.

Bar: as for every attention check (max-abs 2e-3, relative L2 1e-3 against dense float64
attention over the window and the noise block).  The stored keys agree: every level is
exact in F16, the turn changes k[63] by under a quarter of its F16 step, and its q8_0
block (k[63] the only nonzero value) gets the exact scale j / 16 and code +-127 on both
sides; the small turned k[127] may differ by one F16 or q8_0 step, ~1e-6 in a score.  The
query's k[63] weight rounds to 7.375 in F16 on the GPU (the oracle keeps 7.3749).
"""

import numpy as np
import pytest
import torch

import synth
from oracle import ring_oracle as orc
from speculative_decoding_draft_kv_gb300 import ring as R
from tests.ring_harness import assert_close

pytestmark = pytest.mark.gpu

HEAD_DIM, N_HEAD_KV, N_HEAD, Q_LEN, THETA = 128, 8, 32, 8, 1e6
KV_ROW = N_HEAD_KV * HEAD_DIM
LEVEL = 127.0 / 16.0    # key staircase step: 7.375 * 7.9375 / sqrt(128) * log2(e) = 7.46
Q_AMP = 7.375


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_draft_kv_gb300 import build
    build.build()
    R.library()
    torch.cuda.init()


class RampRows:
    """Pre-RoPE F16 rows by absolute position: K zero but for the staircase in dimension 63
    of every head (level j of `run` positions from p0 on, clipped to -16 .. 16), V the
    seeded synthetic rows."""

    def __init__(self, seed, p0, run, sigma):
        self.seed, self.p0, self.run, self.sigma = seed, p0, run, sigma

    def rows(self, seq, layer, pos):
        pos = np.asarray(pos, np.int64)
        k = np.zeros((len(pos), KV_ROW), np.float16)
        level = np.clip(np.floor_divide(pos - self.p0, self.run), -16, 16)
        ramp = (LEVEL * level).astype(np.float16)                 # exact: 127 j / 16
        for g in range(N_HEAD_KV):
            k[:, g * HEAD_DIM + 63] = ramp
        _, v = synth.context_rows(self.seed, seq, layer, torch.as_tensor(pos), KV_ROW, self.sigma)
        return k, v.numpy()

    def fn(self, seq, layer):
        return lambda pos: self.rows(seq, layer, pos)


def queries(n_seq):
    """Query rows: +-Q_AMP in dimension 63, the sign alternating with the query head."""
    q = np.zeros((n_seq, Q_LEN, N_HEAD, HEAD_DIM), np.float32)
    for h in range(N_HEAD):
        q[:, :, h, 63] = Q_AMP if h % 2 == 0 else -Q_AMP
    return q


@pytest.mark.parametrize("n_seq,cap,kv_format", [
    (1, 4096, "f16"),       # few (sequence, kv head) pairs: the cluster instance
    (1, 4096, "q8_0"),
    (16, 1024, "f16"),      # many pairs: the plain instance (exact running maximum)
    (16, 1024, "q8_0"),     # plain q8_0 instance (lazy reference)
])
def test_scores_far_beyond_one_exponent_range(n_seq, cap, kv_format):
    w = synth.workload(2)
    n_layer = 2
    swa = cap // 2
    # the window's centre after the last step: the staircase crosses zero there
    steps = [cap + 100, cap + 103]
    src = RampRows(w.seed, steps[-1] - cap // 2, cap // 32, w.sigma)
    ring = R.Ring(cap, Q_LEN, HEAD_DIM, N_HEAD_KV, N_HEAD, n_layer, THETA, n_seq=n_seq,
                  swa_window=swa, kv_format=kv_format)
    try:
        for c in steps:
            starts, counts = [], []
            for s in range(n_seq):
                st, nn = ring.rows_needed(s, c)
                starts.append(st)
                counts.append(nn)
            n_rows = sum(counts)
            row_off = np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int64)
            k_rows = np.zeros((n_layer, n_rows, KV_ROW), np.float16)
            v_rows = np.zeros_like(k_rows)
            for s in range(n_seq):
                pos = np.arange(starts[s], c)
                for layer in range(n_layer):
                    k, v = src.rows(s, layer, pos)
                    k_rows[layer, row_off[s]:row_off[s] + counts[s]] = k
                    v_rows[layer, row_off[s]:row_off[s] + counts[s]] = v
            ring.begin_step([c] * n_seq, torch.from_numpy(k_rows).cuda(), torch.from_numpy(v_rows).cuda(),
                            row_off, starts)
        q = queries(n_seq)
        kn = np.zeros((n_seq, Q_LEN, KV_ROW), np.float16)
        vn = np.stack([synth.noise_rows(w.seed, 7, s, 0, Q_LEN, KV_ROW, w.sigma)[1].numpy()
                       for s in range(n_seq)])
        for layer in range(n_layer):
            for kind in ("full", "swa"):
                o = torch.empty((n_seq, Q_LEN, N_HEAD, HEAD_DIM), device="cuda")
                ring.attend(layer, kind, torch.from_numpy(q).cuda(), torch.from_numpy(kn).cuda(),
                            torch.from_numpy(vn).cuda(), o)
                torch.cuda.synchronize()
                got = o.cpu().numpy()
                assert np.isfinite(got).all()
                for s in sorted({0, n_seq - 1}):
                    want = orc.attend_dense(steps[-1], cap, src.fn(s, layer), q[s], kn[s], vn[s],
                                            HEAD_DIM, N_HEAD_KV, N_HEAD, THETA, kind=kind,
                                            swa_window=swa, kv_format=kv_format)
                    assert_close(got[s], want, f"seq {s} layer {layer} {kind} {kv_format}")
        assert ring.device_error() == 0
    finally:
        ring.close()
