"""Float64 CPU oracle of the DFlash draft-KV ring step (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import this package.  It holds no CUDA code and never calls the
library under test.
"""

from .ring_oracle import (  # noqa: F401
    NEG_INF,
    NaiveRollOracle,
    RingOracle,
    align_up,
    attend_dense,
    geometry,
    kv_head_of,
    slot_of,
    softmax_scale,
    masked_attention,
    rope_inv_freq,
    rope_neox,
    rope_rows,
    step_window,
    swa_low,
    to_f16,
)
