"""The five synthetic ring workloads and their commit schedules.

A schedule is the sequence of ``committed`` values (one per sequence) handed to
``ring_begin_step``.  Step sizes are drawn here from seeded numpy generators; how the
ring turns a commit into slots, masks and attention is not this module's business.

The acceptance histogram that drives the steady-state appends is the share of
verifications by accepted draft count printed on the page "speculative : capped
recurrent planes for DFlash" (section "Why the layout matters": uncapped, n-max 7,
1422 verifications).  A step that accepts ``a`` draft tokens commits ``a + 1`` tokens
(the accepted ones plus the target's own token).
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

ACCEPT_HISTOGRAM = {0: 24.5, 1: 19.5, 2: 15.0, 3: 9.9, 4: 7.7, 5: 5.0, 6: 3.6, 7: 14.7}


@dataclass(frozen=True)
class Workload:
    name: str
    cap: int
    q_len: int = 8
    head_dim: int = 128
    n_head_kv: int = 8
    n_head: int = 32
    n_layer: int = 5
    rope_theta: float = 1.0e6
    n_seq: int = 1
    swa_window: int = 0
    sigma: float = 0.5
    steps: int = 1
    seed: int = 0
    kind: str = "decode"          # decode | tiny | bulk | batched | large
    extra: dict = field(default_factory=dict)

    @property
    def kv_row(self) -> int:
        return self.head_dim * self.n_head_kv


WORKLOADS = {
    1: Workload("tiny_ring_cap64_s1_l1", cap=64, n_layer=1, n_seq=1, steps=40,
                seed=0xD17A0001, kind="tiny"),
    2: Workload("steady_decode_cap4096_s1_l5", cap=4096, n_layer=5, n_seq=1, steps=2000,
                seed=0xD17A0002, kind="decode", extra={"prefill": 8192}),
    3: Workload("bulk_stress_cap4096_s1_l5", cap=4096, n_layer=5, n_seq=1, steps=200,
                seed=0xD17A0003, kind="bulk", extra={"jump_max": 30000, "fold_max": 18,
                                                     "p_jump": 0.25}),
    4: Workload("batched_cap4096_s64_l5", cap=4096, n_layer=5, n_seq=64, steps=500,
                swa_window=2048, seed=0xD17A0004, kind="batched",
                extra={"c0_max": 131072}),
    5: Workload("large_ring_cap32768_s16_l5", cap=32768, n_layer=5, n_seq=16, steps=1000,
                seed=0xD17A0005, kind="large", extra={"c0_base": 131072, "c0_spread": 4096}),
}


def workload(k: int, **overrides) -> Workload:
    w = WORKLOADS[k]
    return replace(w, **overrides) if overrides else w


def _accept_draws(rng: np.random.Generator, shape) -> np.ndarray:
    keys = np.array(sorted(ACCEPT_HISTOGRAM), dtype=np.int64)
    p = np.array([ACCEPT_HISTOGRAM[k] for k in keys], dtype=np.float64)
    p = p / p.sum()
    return rng.choice(keys, size=shape, p=p)


def commit_schedule(w: Workload, n_steps: int | None = None) -> np.ndarray:
    """int64 ``[n_calls, n_seq]``: the ``committed`` argument of each begin-step call.

    Row 0 is the first call.  For workloads that start from a long prompt, row 0 is
    the prefill commit (served by the bulk path) and ``n_steps`` decode steps follow.
    """
    n = w.steps if n_steps is None else n_steps
    rng = np.random.default_rng(w.seed ^ 0x5EED5EED)
    S = w.n_seq
    if w.kind == "tiny":
        # each step accepts k in {0..8} uniformly and commits k + 1 rows
        inc = rng.integers(0, 9, size=(n, S)) + 1
        return np.cumsum(inc, axis=0).astype(np.int64)
    if w.kind == "decode":
        c0 = np.full((1, S), w.extra["prefill"], dtype=np.int64)
        inc = _accept_draws(rng, (n, S)) + 1
        return np.concatenate([c0, c0 + np.cumsum(inc, axis=0)], axis=0)
    if w.kind == "bulk":
        out = []
        c = np.zeros(S, dtype=np.int64)
        for t in range(n):
            if t == 0 or rng.random() < w.extra["p_jump"]:
                c = c + rng.integers(1, w.extra["jump_max"] + 1, size=S)
            else:
                c = c + rng.integers(1, w.extra["fold_max"] + 1, size=S)
            out.append(c.copy())
        return np.stack(out).astype(np.int64)
    if w.kind == "batched":
        c0 = rng.integers(1, w.extra["c0_max"] + 1, size=(1, S)).astype(np.int64)
        inc = _accept_draws(rng, (n, S)) + 1
        return np.concatenate([c0, c0 + np.cumsum(inc, axis=0)], axis=0)
    if w.kind == "large":
        c0 = (w.extra["c0_base"] + rng.integers(0, w.extra["c0_spread"], size=(1, S))).astype(np.int64)
        inc = _accept_draws(rng, (n, S)) + 1
        return np.concatenate([c0, c0 + np.cumsum(inc, axis=0)], axis=0)
    raise ValueError(f"unknown workload kind {w.kind!r}")
