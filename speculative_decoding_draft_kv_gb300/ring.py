"""Thin Python binding of the C ABI declared in ``include/dflash_ring.h``.

Every function here has the name of the C entry point it calls and does nothing but
marshal arguments (tensor pointers, shapes, the current CUDA stream) and turn a
negative status into :class:`RingError`.  All computation happens in the CUDA library;
if that library has not been built, loading fails loudly -- there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libdflash_ring.so")

RING_OK = 0
RING_EINVAL = -1
RING_ERANGE = -2
RING_ENOMEM = -3
RING_ECUDA = -4
RING_ESTATE = -5
RING_EDEVICE = -6
RING_MASK_FULL = 0
RING_MASK_SWA = 1
RING_KV_F16 = 0
RING_KV_Q8_0 = 1
KV_FORMATS = {"f16": RING_KV_F16, "q8_0": RING_KV_Q8_0}
MASK_KINDS = {"full": RING_MASK_FULL, "swa": RING_MASK_SWA}

# C symbols the header declares (checked by the test-suite against the shared object).
EXPORTED = (
    "ring_init", "ring_init_ex", "ring_destroy", "ring_get_geometry", "ring_rows_needed",
    "ring_begin_step", "ring_attend", "ring_step", "ring_get_slot_pos", "ring_get_mask",
    "ring_get_tile_flags", "ring_get_kv", "ring_device_error", "ring_describe",
    "ring_profile_enable", "ring_profile_read", "ring_launch_count", "ring_attend_static",
    "ring_last_error", "ring_set_producer", "ring_begin_step_features", "ring_recompute_window",
    "ring_draft_step", "ring_get_kv_q8", "ring_clock_enable", "ring_clock_read",
    "ring_check_bounded_wait", "ring_attend_static_device_error",
)


class RingError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code


class RingParams(ctypes.Structure):
    _fields_ = [("cap", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_head_kv", ctypes.c_int32),
                ("n_head", ctypes.c_int32), ("n_layer", ctypes.c_int32),
                ("rope_theta", ctypes.c_float), ("n_seq", ctypes.c_int32),
                ("swa_window", ctypes.c_int32), ("bulk_chunk", ctypes.c_int32),
                ("tiles_per_split", ctypes.c_int32), ("max_cluster", ctypes.c_int32),
                ("kv_format", ctypes.c_int32), ("step_split", ctypes.c_int32)]


class RingGeometry(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "cap", "q_len", "a_step", "trash_slot", "kv_total", "kv_row", "head_dim", "n_head_kv",
        "n_head", "n_layer", "n_seq", "swa_window", "bulk_chunk", "tile_slots", "n_tiles",
        "tiles_per_split", "n_splits", "cluster", "groups")] + [("cache_bytes", ctypes.c_int64),
                                           ("device_bytes", ctypes.c_int64),
                                           ("step_split", ctypes.c_int32),
                                           ("step_ctas", ctypes.c_int32)]


class RingAttendStaticArgs(ctypes.Structure):
    _fields_ = [("cap", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_head_kv", ctypes.c_int32),
                ("n_head", ctypes.c_int32), ("n_seq", ctypes.c_int32),
                ("rope_theta", ctypes.c_float),
                ("committed", ctypes.POINTER(ctypes.c_int64)),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("mask", ctypes.c_void_p),
                ("q", ctypes.c_void_p), ("k_noise", ctypes.c_void_p),
                ("v_noise", ctypes.c_void_p), ("o", ctypes.c_void_p)]


class RingProfile(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int64 * 6), ("total_ms", ctypes.c_double * 6)]


class RingProducer(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("eps", ctypes.c_float), ("wk", ctypes.c_void_p),
                ("wv", ctypes.c_void_p), ("k_norm", ctypes.c_void_p), ("wq", ctypes.c_void_p),
                ("q_norm", ctypes.c_void_p)]


PROFILE_CLASSES = ("bulk", "begin", "attend", "combine", "step_graph", "produce")

_LIB = None
_N_SEQ = {}      # handle -> n_seq, so per-step calls skip a geometry query


def _load():
    global _LIB
    if _LIB is not None:
        return _LIB
    path = os.environ.get("DFLASH_RING_LIB", LIB_PATH)
    if not os.path.exists(path):
        raise RuntimeError(
            f"the CUDA ring library is not built ({path} missing); run "
            "`python -c 'import __graft_entry__ as g; g.build()'` first")
    L = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    p64 = ctypes.POINTER(ctypes.c_int64)
    sig = {
        "ring_init": ([ctypes.POINTER(vp), i32, i32, i32, i32, i32, i32, ctypes.c_float], ctypes.c_int),
        "ring_init_ex": ([ctypes.POINTER(vp), ctypes.POINTER(RingParams)], ctypes.c_int),
        "ring_destroy": ([vp], ctypes.c_int),
        "ring_get_geometry": ([vp, ctypes.POINTER(RingGeometry)], ctypes.c_int),
        "ring_rows_needed": ([vp, i32, i64, p64, ctypes.POINTER(i32)], ctypes.c_int),
        "ring_begin_step": ([vp, p64, vp, vp, p64, p64, i64, vp], ctypes.c_int),
        "ring_attend": ([vp, i32, i32, vp, vp, vp, vp, vp], ctypes.c_int),
        "ring_step": ([vp, p64, vp, vp, p64, p64, i64, i32, ctypes.POINTER(vp), ctypes.POINTER(vp),
                       ctypes.POINTER(vp), ctypes.POINTER(vp), vp], ctypes.c_int),
        "ring_get_slot_pos": ([vp, i32, vp], ctypes.c_int),
        "ring_get_mask": ([vp, i32, i32, vp], ctypes.c_int),
        "ring_get_tile_flags": ([vp, i32, i32, vp], ctypes.c_int),
        "ring_get_kv": ([vp, i32, i32, vp, vp], ctypes.c_int),
        "ring_get_kv_q8": ([vp, i32, i32, vp, vp, vp, vp], ctypes.c_int),
        "ring_device_error": ([vp, ctypes.POINTER(ctypes.c_uint32)], ctypes.c_int),
        "ring_describe": ([vp, ctypes.c_char_p, ctypes.c_size_t], ctypes.c_int),
        "ring_profile_enable": ([vp, i32], ctypes.c_int),
        "ring_profile_read": ([vp, ctypes.POINTER(RingProfile)], ctypes.c_int),
        "ring_launch_count": ([vp], ctypes.c_int64),
        "ring_attend_static": ([ctypes.POINTER(RingAttendStaticArgs), vp], ctypes.c_int),
        "ring_last_error": ([vp], ctypes.c_char_p),
        "ring_set_producer": ([vp, ctypes.POINTER(RingProducer)], ctypes.c_int),
        "ring_begin_step_features": ([vp, p64, vp, p64, p64, i64, vp], ctypes.c_int),
        "ring_recompute_window": ([vp, p64, vp, p64, p64, i64, vp], ctypes.c_int),
        "ring_draft_step": ([vp, p64, vp, p64, p64, i64, vp, ctypes.POINTER(i32),
                             ctypes.POINTER(vp), vp], ctypes.c_int),
        "ring_clock_enable": ([vp, i32], ctypes.c_int),
        "ring_clock_read": ([vp, i32, ctypes.POINTER(ctypes.c_double), p64], ctypes.c_int),
        "ring_check_bounded_wait": ([vp, i32, i32, vp], ctypes.c_int),
        "ring_attend_static_device_error": ([ctypes.POINTER(ctypes.c_uint32)], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _LIB = L
    return L


def library():
    """The loaded ``ctypes.CDLL`` (loads it on first use)."""
    return _load()


def ring_last_error(h) -> str:
    return _load().ring_last_error(h).decode()


def _check(rc: int, h, what: str):
    if rc != RING_OK:
        raise RingError(rc, f"{what}: {ring_last_error(h)}")


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _dev_ptr(t, dtype, name):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _i64_array(vals, n, name):
    a = np.ascontiguousarray(np.asarray(vals, dtype=np.int64).reshape(-1))
    if a.size != n:
        raise ValueError(f"{name} must have {n} entries, got {a.size}")
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def ring_init(cap, q_len, head_dim, n_head_kv, n_head, n_layer, rope_theta):
    h = ctypes.c_void_p()
    rc = _load().ring_init(ctypes.byref(h), cap, q_len, head_dim, n_head_kv, n_head, n_layer,
                           float(rope_theta))
    _check(rc, None, "ring_init")
    _N_SEQ[h.value] = 1
    return h


def ring_init_ex(cap, q_len, head_dim, n_head_kv, n_head, n_layer, rope_theta, n_seq=1,
                 swa_window=0, bulk_chunk=0, tiles_per_split=0, max_cluster=0, kv_format="f16",
                 step_split=0):
    p = RingParams(cap, q_len, head_dim, n_head_kv, n_head, n_layer, float(rope_theta), n_seq,
                   swa_window, bulk_chunk, tiles_per_split, max_cluster,
                   KV_FORMATS.get(kv_format, kv_format), step_split)
    h = ctypes.c_void_p()
    rc = _load().ring_init_ex(ctypes.byref(h), ctypes.byref(p))
    _check(rc, None, "ring_init_ex")
    _N_SEQ[h.value] = max(1, int(n_seq))
    return h


def ring_destroy(h):
    if h:
        _N_SEQ.pop(getattr(h, "value", h), None)
        _load().ring_destroy(h)


def ring_get_geometry(h) -> dict:
    g = RingGeometry()
    _check(_load().ring_get_geometry(h, ctypes.byref(g)), h, "ring_get_geometry")
    return {name: getattr(g, name) for name, _ in RingGeometry._fields_}


def ring_rows_needed(h, seq, committed):
    start = ctypes.c_int64()
    n_new = ctypes.c_int32()
    _check(_load().ring_rows_needed(h, seq, int(committed), ctypes.byref(start), ctypes.byref(n_new)),
           h, "ring_rows_needed")
    return start.value, n_new.value


def ring_begin_step(h, committed, k_rows, v_rows, row_off, first_pos, stream=None):
    """``k_rows``/``v_rows``: CUDA float16 [n_layer, n_rows, kv_row] or None."""
    import torch
    n_seq = _N_SEQ.get(getattr(h, "value", h)) or ring_get_geometry(h)["n_seq"]
    c_arr, c_ptr = _i64_array(committed, n_seq, "committed")
    o_arr, o_ptr = _i64_array(row_off, n_seq, "row_off")
    f_arr, f_ptr = _i64_array(first_pos, n_seq, "first_pos")
    n_rows = 0 if k_rows is None else int(k_rows.shape[1])
    if k_rows is not None and (k_rows.shape != v_rows.shape or k_rows.dim() != 3):
        raise ValueError("k_rows and v_rows must both be [n_layer, n_rows, kv_row]")
    rc = _load().ring_begin_step(h, c_ptr, _dev_ptr(k_rows, torch.float16, "k_rows"),
                                 _dev_ptr(v_rows, torch.float16, "v_rows"), o_ptr, f_ptr,
                                 n_rows, _stream(stream))
    _check(rc, h, "ring_begin_step")


def ring_set_producer(h, hidden, eps, wk, wv, k_norm, wq=None, q_norm=None):
    """wk, wv: CUDA float16 [n_layer, kv_row, hidden]; k_norm: CUDA float32
    [n_layer, head_dim]; optional wq (float16 [n_layer, n_head * head_dim, hidden]) and
    q_norm (float32 [n_layer, head_dim]) for ring_draft_step.  The ring copies them
    (synchronously); all None detaches the producer."""
    import torch
    if wk is None and wv is None and k_norm is None:
        _check(_load().ring_set_producer(h, None), h, "ring_set_producer")
        return
    p = RingProducer(int(hidden), float(eps), _dev_ptr(wk, torch.float16, "wk"),
                     _dev_ptr(wv, torch.float16, "wv"), _dev_ptr(k_norm, torch.float32, "k_norm"),
                     _dev_ptr(wq, torch.float16, "wq"), _dev_ptr(q_norm, torch.float32, "q_norm"))
    _check(_load().ring_set_producer(h, ctypes.byref(p)), h, "ring_set_producer")


def ring_begin_step_features(h, committed, feat, row_off, first_pos, stream=None,
                             _entry="ring_begin_step_features"):
    """``feat``: CUDA float16 [n_rows, hidden] or None (no sequence appends)."""
    import torch
    n_seq = _N_SEQ.get(getattr(h, "value", h)) or ring_get_geometry(h)["n_seq"]
    c_arr, c_ptr = _i64_array(committed, n_seq, "committed")
    o_arr, o_ptr = _i64_array(row_off, n_seq, "row_off")
    f_arr, f_ptr = _i64_array(first_pos, n_seq, "first_pos")
    n_rows = 0 if feat is None else int(feat.shape[0])
    if feat is not None and feat.dim() != 2:
        raise ValueError("feat must be [n_rows, hidden]")
    rc = getattr(_load(), _entry)(h, c_ptr, _dev_ptr(feat, torch.float16, "feat"), o_ptr, f_ptr,
                                  n_rows, _stream(stream))
    _check(rc, h, _entry)


def ring_draft_step(h, committed, feat, row_off, first_pos, noise_h, mask_kinds, o, stream=None):
    """``noise_h``: CUDA float16 [n_layer, n_seq, q_len, hidden]; ``mask_kinds``: one
    "full"/"swa" (or code) per layer; ``o``: n_layer CUDA float32 tensors
    [n_seq, q_len, n_head, head_dim]."""
    import torch
    n_seq = _N_SEQ.get(getattr(h, "value", h)) or ring_get_geometry(h)["n_seq"]
    c_arr, c_ptr = _i64_array(committed, n_seq, "committed")
    o_arr, o_ptr = _i64_array(row_off, n_seq, "row_off")
    f_arr, f_ptr = _i64_array(first_pos, n_seq, "first_pos")
    n_rows = 0 if feat is None else int(feat.shape[0])
    kinds = np.ascontiguousarray([MASK_KINDS.get(k, k) for k in mask_kinds], dtype=np.int32)
    arr = ctypes.c_void_p * len(o)
    op = arr(*[_dev_ptr(t, torch.float32, "o").value for t in o])
    rc = _load().ring_draft_step(h, c_ptr, _dev_ptr(feat, torch.float16, "feat"), o_ptr, f_ptr,
                                 n_rows, _dev_ptr(noise_h, torch.float16, "noise_h"),
                                 kinds.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), op,
                                 _stream(stream))
    _check(rc, h, "ring_draft_step")


def ring_recompute_window(h, committed, feat, row_off, first_pos, stream=None):
    """Every row of [lo, committed) produced again from ``feat`` (rows covering it)."""
    ring_begin_step_features(h, committed, feat, row_off, first_pos, stream,
                             _entry="ring_recompute_window")


def ring_attend(h, layer, mask_kind, q, k_noise, v_noise, o, stream=None):
    """q, o: CUDA float32 [n_seq, q_len, n_head, head_dim]; noise: float16 [n_seq, q_len, kv_row]."""
    import torch
    kind = MASK_KINDS.get(mask_kind, mask_kind)
    rc = _load().ring_attend(h, layer, kind, _dev_ptr(q, torch.float32, "q"),
                             _dev_ptr(k_noise, torch.float16, "k_noise"),
                             _dev_ptr(v_noise, torch.float16, "v_noise"),
                             _dev_ptr(o, torch.float32, "o"), _stream(stream))
    _check(rc, h, "ring_attend")


def ring_step(h, committed, k_rows, v_rows, row_off, first_pos, mask_kind, q, k_noise, v_noise,
              o, stream=None):
    """One begin_step plus every layer's attention, replayed as one CUDA graph.

    ``q``, ``k_noise``, ``v_noise``, ``o``: sequences of n_layer CUDA tensors (layouts as
    for :func:`ring_attend`); ``k_rows``/``v_rows`` as for :func:`ring_begin_step`.
    """
    import torch
    n_seq = _N_SEQ.get(getattr(h, "value", h)) or ring_get_geometry(h)["n_seq"]
    c_arr, c_ptr = _i64_array(committed, n_seq, "committed")
    o_arr, o_ptr = _i64_array(row_off, n_seq, "row_off")
    f_arr, f_ptr = _i64_array(first_pos, n_seq, "first_pos")
    n_rows = 0 if k_rows is None else int(k_rows.shape[1])
    n_layer = len(q)
    arr = ctypes.c_void_p * n_layer
    qp = arr(*[_dev_ptr(t, torch.float32, "q").value for t in q])
    kp = arr(*[_dev_ptr(t, torch.float16, "k_noise").value for t in k_noise])
    vp_ = arr(*[_dev_ptr(t, torch.float16, "v_noise").value for t in v_noise])
    op = arr(*[_dev_ptr(t, torch.float32, "o").value for t in o])
    kind = MASK_KINDS.get(mask_kind, mask_kind)
    rc = _load().ring_step(h, c_ptr, _dev_ptr(k_rows, torch.float16, "k_rows"),
                           _dev_ptr(v_rows, torch.float16, "v_rows"), o_ptr, f_ptr, n_rows, kind,
                           qp, kp, vp_, op, _stream(stream))
    _check(rc, h, "ring_step")


def ring_get_slot_pos(h, seq) -> np.ndarray:
    g = ring_get_geometry(h)
    out = np.empty(g["cap"], np.int32)
    _check(_load().ring_get_slot_pos(h, seq, out.ctypes.data_as(ctypes.c_void_p)), h,
           "ring_get_slot_pos")
    return out


def ring_get_mask(h, seq, mask_kind) -> np.ndarray:
    g = ring_get_geometry(h)
    out = np.empty((g["q_len"], g["kv_total"]), np.float32)
    kind = MASK_KINDS.get(mask_kind, mask_kind)
    _check(_load().ring_get_mask(h, seq, kind, out.ctypes.data_as(ctypes.c_void_p)), h,
           "ring_get_mask")
    return out


def ring_get_tile_flags(h, seq, mask_kind) -> np.ndarray:
    g = ring_get_geometry(h)
    out = np.empty(g["n_tiles"], np.uint8)
    kind = MASK_KINDS.get(mask_kind, mask_kind)
    _check(_load().ring_get_tile_flags(h, seq, kind, out.ctypes.data_as(ctypes.c_void_p)), h,
           "ring_get_tile_flags")
    return out


def ring_get_kv(h, seq, layer):
    """(K, V) as float16 numpy arrays [kv_total, kv_row] (the page's row layout)."""
    g = ring_get_geometry(h)
    k = np.empty((g["kv_total"], g["kv_row"]), np.uint16)
    v = np.empty_like(k)
    _check(_load().ring_get_kv(h, seq, layer, k.ctypes.data_as(ctypes.c_void_p),
                               v.ctypes.data_as(ctypes.c_void_p)), h, "ring_get_kv")
    return k.view(np.float16), v.view(np.float16)


def ring_get_kv_q8(h, seq, layer):
    """q8_0 rings: (K codes int8 [kv_total, kv_row], K scales float16 [kv_total, kv_row/32],
    V codes, V scales) in the page's row layout."""
    g = ring_get_geometry(h)
    kc = np.empty((g["kv_total"], g["kv_row"]), np.int8)
    vc = np.empty_like(kc)
    ks = np.empty((g["kv_total"], g["kv_row"] // 32), np.uint16)
    vs = np.empty_like(ks)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check(_load().ring_get_kv_q8(h, seq, layer, ptr(kc), ptr(ks), ptr(vc), ptr(vs)), h,
           "ring_get_kv_q8")
    return kc, ks.view(np.float16), vc, vs.view(np.float16)


def ring_device_error(h) -> int:
    bits = ctypes.c_uint32()
    rc = _load().ring_device_error(h, ctypes.byref(bits))
    if rc not in (RING_OK, RING_EDEVICE):
        _check(rc, h, "ring_device_error")
    return bits.value


def ring_describe(h) -> str:
    buf = ctypes.create_string_buffer(256)
    _check(_load().ring_describe(h, buf, 256), h, "ring_describe")
    return buf.value.decode()


def ring_profile_enable(h, on=True):
    _check(_load().ring_profile_enable(h, 1 if on else 0), h, "ring_profile_enable")


def ring_profile_read(h) -> dict:
    p = RingProfile()
    _check(_load().ring_profile_read(h, ctypes.byref(p)), h, "ring_profile_read")
    return {name: {"launches": p.launches[i], "total_ms": p.total_ms[i]}
            for i, name in enumerate(PROFILE_CLASSES)}


def ring_launch_count(h) -> int:
    return int(_load().ring_launch_count(h))


def ring_clock_enable(h, on=True):
    _check(_load().ring_clock_enable(h, 1 if on else 0), h, "ring_clock_enable")


CLOCK_KINDS = {"attend": 0, "produce": 1, "project": 2}


def ring_clock_read(h, kind="attend"):
    """(summed milliseconds, launches) of one kernel kind since the last read: "attend"
    (attention), "produce" (context-row producer) or "project" (noise projections)."""
    ms = ctypes.c_double()
    n = ctypes.c_int64()
    _check(_load().ring_clock_read(h, CLOCK_KINDS[kind], ctypes.byref(ms), ctypes.byref(n)), h,
           "ring_clock_read")
    return ms.value, n.value


def ring_check_bounded_wait(h, which, limit_us, stream=None):
    """Launch the bounded-wait self-test kernel (0: mbarrier, 1: cross-CTA counter)."""
    _check(_load().ring_check_bounded_wait(h, int(which), int(limit_us), _stream(stream)), h,
           "ring_check_bounded_wait")


def ring_attend_static_device_error() -> int:
    """Read and clear ring_attend_static's device error word on the current device."""
    bits = ctypes.c_uint32()
    rc = _load().ring_attend_static_device_error(ctypes.byref(bits))
    if rc not in (RING_OK, RING_EDEVICE):
        _check(rc, None, "ring_attend_static_device_error")
    return bits.value


def ring_attend_static(cap, q_len, n_head_kv, n_head, rope_theta, committed, k, v, mask, q,
                       k_noise, v_noise, o, head_dim=128, stream=None):
    """One layer's attention over caller-owned buffers, allocating nothing.

    k, v: CUDA float16 [n_seq, n_head_kv, kv_total, head_dim] (noise rows written back);
    mask: CUDA float32 [n_seq, q_len, kv_total]; q, o: CUDA float32
    [n_seq, q_len, n_head, head_dim]; noise rows: CUDA float16 [n_seq, q_len, kv_row].
    """
    import torch
    n_seq = int(q.shape[0])
    c_arr, c_ptr = _i64_array(committed, n_seq, "committed")
    args = RingAttendStaticArgs(cap, q_len, head_dim, n_head_kv, n_head, n_seq, float(rope_theta),
                                c_ptr, _dev_ptr(k, torch.float16, "k"), _dev_ptr(v, torch.float16, "v"),
                                _dev_ptr(mask, torch.float32, "mask"), _dev_ptr(q, torch.float32, "q"),
                                _dev_ptr(k_noise, torch.float16, "k_noise"),
                                _dev_ptr(v_noise, torch.float16, "v_noise"),
                                _dev_ptr(o, torch.float32, "o"))
    _check(_load().ring_attend_static(ctypes.byref(args), _stream(stream)), None,
           "ring_attend_static")


class Ring:
    """Owning handle around the C entry points (closes itself)."""

    def __init__(self, cap, q_len, head_dim, n_head_kv, n_head, n_layer, rope_theta, n_seq=1,
                 swa_window=0, bulk_chunk=0, tiles_per_split=0, max_cluster=0, kv_format="f16",
                 step_split=0):
        self.h = ring_init_ex(cap, q_len, head_dim, n_head_kv, n_head, n_layer, rope_theta,
                              n_seq, swa_window, bulk_chunk, tiles_per_split, max_cluster,
                              kv_format, step_split)
        self.geometry = ring_get_geometry(self.h)

    def rows_needed(self, seq, committed):
        return ring_rows_needed(self.h, seq, committed)

    def begin_step(self, committed, k_rows, v_rows, row_off, first_pos, stream=None):
        ring_begin_step(self.h, committed, k_rows, v_rows, row_off, first_pos, stream)

    def set_producer(self, hidden, eps, wk, wv, k_norm, wq=None, q_norm=None):
        ring_set_producer(self.h, hidden, eps, wk, wv, k_norm, wq, q_norm)

    def draft_step(self, committed, feat, row_off, first_pos, noise_h, mask_kinds, o,
                   stream=None):
        ring_draft_step(self.h, committed, feat, row_off, first_pos, noise_h, mask_kinds, o,
                        stream)

    def begin_step_features(self, committed, feat, row_off, first_pos, stream=None):
        ring_begin_step_features(self.h, committed, feat, row_off, first_pos, stream)

    def recompute_window(self, committed, feat, row_off, first_pos, stream=None):
        ring_recompute_window(self.h, committed, feat, row_off, first_pos, stream)

    def attend(self, layer, mask_kind, q, k_noise, v_noise, o, stream=None):
        ring_attend(self.h, layer, mask_kind, q, k_noise, v_noise, o, stream)

    def step(self, committed, k_rows, v_rows, row_off, first_pos, mask_kind, q, k_noise, v_noise,
             o, stream=None):
        ring_step(self.h, committed, k_rows, v_rows, row_off, first_pos, mask_kind, q, k_noise,
                  v_noise, o, stream)

    def slot_pos(self, seq=0):
        return ring_get_slot_pos(self.h, seq)

    def mask(self, seq=0, kind="full"):
        return ring_get_mask(self.h, seq, kind)

    def tile_flags(self, seq=0, kind="full"):
        return ring_get_tile_flags(self.h, seq, kind)

    def kv(self, seq, layer):
        return ring_get_kv(self.h, seq, layer)

    def kv_q8(self, seq, layer):
        return ring_get_kv_q8(self.h, seq, layer)

    def device_error(self):
        return ring_device_error(self.h)

    def describe(self):
        return ring_describe(self.h)

    def launch_count(self):
        return ring_launch_count(self.h)

    def clock_enable(self, on=True):
        ring_clock_enable(self.h, on)

    def clock_read(self, kind="attend"):
        return ring_clock_read(self.h, kind)

    def check_bounded_wait(self, which, limit_us, stream=None):
        ring_check_bounded_wait(self.h, which, limit_us, stream)

    def close(self):
        if self.h:
            ring_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
