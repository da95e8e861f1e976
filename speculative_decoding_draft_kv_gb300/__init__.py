"""DFlash draft-KV ring step for one GB300 GPU (sm_103a).

The computation lives in the CUDA library ``_lib/libdflash_ring.so`` behind the C ABI of
``include/dflash_ring.h``; :mod:`.ring` is the thin binding with the same names, and
:mod:`.build` compiles the library.  Importing this package does not load the library;
the first call into :mod:`.ring` does, and fails loudly if it was not built.
"""

from .ring import (  # noqa: F401
    EXPORTED,
    MASK_KINDS,
    RING_MASK_FULL,
    RING_MASK_SWA,
    Ring,
    RingError,
    ring_attend,
    ring_attend_static,
    ring_begin_step,
    ring_begin_step_features,
    ring_describe,
    ring_destroy,
    ring_device_error,
    ring_draft_step,
    ring_get_geometry,
    ring_get_kv,
    ring_get_kv_q8,
    ring_get_mask,
    ring_get_slot_pos,
    ring_get_tile_flags,
    ring_init,
    ring_init_ex,
    ring_last_error,
    ring_launch_count,
    ring_recompute_window,
    ring_profile_enable,
    ring_profile_read,
    ring_rows_needed,
    ring_set_producer,
    ring_step,
)
