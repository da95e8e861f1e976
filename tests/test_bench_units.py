"""The unit behind bench.py's roofline: the visible K/V rows of one attention launch must be
exactly the slots the oracle's masks open (ring slots inside the window plus the noise
block).  CPU only."""

import numpy as np
import pytest

import bench
import synth
from oracle import ring_oracle as orc


@pytest.mark.parametrize("cap,swa", [(64, 24), (48, 100), (200, 40)])
def test_visible_rows_equal_the_slots_the_masks_open(cap, swa):
    w = synth.workload(1, cap=cap, swa_window=swa)
    r = orc.RingOracle(w.cap, w.q_len, 2, 1, 1, 1, w.rope_theta, swa_window=swa)
    for c in [0, 5, 30, 63, 64, 65, 150, 400]:
        start, n_new = r.rows_needed(c)
        z = np.zeros((1, n_new, 2), np.float16)
        r.begin_step(c, z, z, start)
        for kind in ("full", "swa"):
            opened = int((r.mask(kind) == 0).any(axis=0).sum())
            assert bench.visible_rows(w, [c], kind) == opened, (c, kind)


def test_visible_rows_sum_over_sequences():
    w = synth.workload(1, cap=64, swa_window=24)
    assert bench.visible_rows(w, [0, 10, 100], "full") == (0 + 8) + (10 + 8) + (64 + 8)
    assert bench.visible_rows(w, [0, 10, 100], "swa") == (0 + 8) + (10 + 8) + (24 + 8)


def test_oracle_baseline_spreads_units_over_processes():
    """The oracle leg splits the workload's (sequence, layer) units over host processes,
    at most one per unit, and reports how many it used."""
    import os

    import synth

    w = synth.workload(1, cap=64, n_layer=2, n_seq=2)
    cpu = bench.cpu_baseline(w, "full", n_steps=3)
    assert cpu["kind"] == "oracle" and cpu["value"] > 0
    assert cpu["cores"] == min(os.cpu_count() or 1, 4)
    assert "4 (sequence, layer) units" in cpu["sample"]


def test_tile_flags_of_a_mask():
    import numpy as np
    inf = -np.inf
    m = np.full((2, 130), inf, np.float32)
    m[:, 0:64] = 0          # tile 0: every slot, every row
    m[0, 70] = 0            # tile 1: one slot, one row
    m[:, 128:130] = 0       # tile 2: a ragged two-slot tile, fully visible -> mixed
    np.testing.assert_array_equal(bench._tile_flags(m, 64), [1, 2, 2])
    m[0, 70] = inf
    np.testing.assert_array_equal(bench._tile_flags(m, 64), [1, 0, 2])


def test_code_hash_ignores_comments_and_whitespace_only():
    src = "__global__ void k(int *p) {\n    p[0] = 1;  // one\n}\n"
    same = "/* a kernel */\n__global__  void k(int *p)\n{ p[0] = 1; }\n// end\n"
    other = "__global__ void k(int *p) {\n    p[0] = 2;  // one\n}\n"
    assert bench._code_hash(src) == bench._code_hash(same)
    assert bench._code_hash(src) != bench._code_hash(other)

