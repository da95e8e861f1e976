"""Seeded synthetic inputs for the draft-KV ring step.

This package only draws numbers: counter-based pseudo-random K/V rows, queries,
noise-block rows, fused features and producer weights, plus the per-step commit
schedules of the five ring workloads.  It contains none of the ring's own arithmetic
(no slot map, no projection, no norm, no RoPE, no mask, no attention), so both the CUDA
path and the float64 oracle can take their inputs from it.
"""

from .gen import (  # noqa: F401
    KIND_K_ROW,
    KIND_V_ROW,
    KIND_Q,
    KIND_K_NOISE,
    KIND_V_NOISE,
    hash32,
    gaussian_values,
    context_rows,
    query_block,
    noise_rows,
    feature_rows,
    producer_weights,
    query_weights,
    noise_hidden,
)
from .workloads import (  # noqa: F401
    ACCEPT_HISTOGRAM,
    Workload,
    WORKLOADS,
    workload,
    commit_schedule,
)
