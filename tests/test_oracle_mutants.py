"""Planted mistakes in the oracle must be caught by its pins.

Each mutant patches one decision of the float64 oracle (on the CPU, inside this test
only) with a plausible error -- a dropped term, an off-by-one bound, a wrong index map,
a transposed operand -- and at least one pin of tests/test_oracle_pins.py or
tests/test_oracle_equivalence.py has to fail under it.  This is what makes the pins
worth trusting.
"""

import contextlib

import numpy as np
import pytest

from oracle import ring_oracle as orc
from tests import test_oracle_equivalence as eqv
from tests import test_oracle_pins as pins


def _rope_drop_term(x, pos, theta):
    x = np.asarray(x, np.float64)
    half = x.shape[-1] // 2
    ang = np.asarray(pos, np.float64)[..., None] * orc.rope_inv_freq(x.shape[-1], theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c, x1 * s + x2 * c], axis=-1)


def _rope_gptj_pairs(x, pos, theta):
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    ang = np.asarray(pos, np.float64)[..., None] * orc.rope_inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x1 * c - x2 * s
    out[..., 1::2] = x1 * s + x2 * c
    return out


def _inv_freq_wrong_exponent(head_dim, theta):
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(np.float64(theta), -i / head_dim)


def _to_f16_truncate(x):
    x = np.asarray(x, np.float64).astype(np.float32)
    bits = x.view(np.uint32) & np.uint32(0xFFFFE000)       # chop the low mantissa bits
    return bits.view(np.float32).astype(np.float16)


def _step_window_lo_off_by_one(committed, next_pos, cap):
    win = min(committed, cap)
    lo = committed - win + 1
    start = max(next_pos, lo)
    return win, lo, start, committed - start


def _mask_full_shows_empty_slots(self):
    # On a ring the window test can only reject never-written slots (every written slot
    # already holds a position in [lo, c)), so the plausible slip is to skip it.
    m = np.full((self.q_len, self.kv_total), orc.NEG_INF, np.float32)
    m[:, :self.cap + self.q_len] = 0.0
    return m


def _mask_swa_uses_full_window(self):
    c = self.committed
    lo = c - min(c, self.cap)
    m = np.full((self.q_len, self.kv_total), orc.NEG_INF, np.float32)
    for s in range(self.cap):
        if lo <= self.slot_pos[s] < c:
            m[:, s] = 0.0
    for i in range(self.q_len):
        m[i, self.cap:self.cap + i + 1] = 0.0
    return m


def _mask_swa_not_causal(self):
    c = self.committed
    slo = orc.swa_low(c, self.cap, self.swa_window)
    m = np.full((self.q_len, self.kv_total), orc.NEG_INF, np.float32)
    for s in range(self.cap):
        if slo <= self.slot_pos[s] < c:
            m[:, s] = 0.0
    m[:, self.cap:self.cap + self.q_len] = 0.0
    return m


def _write_noise_shifted(self, layer, k_noise, v_noise):
    c = self.committed
    for j in range(self.q_len):
        kr = orc.rope_rows(k_noise[j], c + j + 1, self.n_head_kv, self.head_dim, self.theta)
        self.k[layer, self.cap + j] = orc.to_f16(kr)
        self.v[layer, self.cap + j] = v_noise[j]


def _masked_attention_kv_swapped(q, k, v, mask, scale):
    return _ORIG_MA(q, v, k, mask, scale)


_ORIG_MA = orc.masked_attention
_ORIG_BEGIN = orc.RingOracle.begin_step


def _begin_step_no_pad_zero(self, committed, k_rows, v_rows, first_pos):
    keep_k = self.k[:, self.trash_slot].copy()
    keep_v = self.v[:, self.trash_slot].copy()
    path = _ORIG_BEGIN(self, committed, k_rows, v_rows, first_pos)
    self.k[:, self.trash_slot] = keep_k
    self.v[:, self.trash_slot] = keep_v
    return path


_ORIG_RMS = orc.rms_norm_heads


def _rms_whole_row(x, w, eps, n_heads, head_dim):
    return _ORIG_RMS(x, np.tile(np.asarray(w, np.float64), n_heads), eps, 1, n_heads * head_dim)


def _rms_eps_outside_root(x, w, eps, n_heads, head_dim):
    x = np.asarray(x, np.float64)
    r = x.reshape(x.shape[:-1] + (n_heads, head_dim))
    ms = np.mean(r * r, axis=-1, keepdims=True)
    return (r / (np.sqrt(ms) + eps) * np.asarray(w, np.float64)).reshape(x.shape)


def _rms_weight_ignored(x, w, eps, n_heads, head_dim):
    return _ORIG_RMS(x, np.ones(head_dim), eps, n_heads, head_dim)


def _rms_mean_over_heads(x, w, eps, n_heads, head_dim):
    x = np.asarray(x, np.float64)
    r = x.reshape(x.shape[:-1] + (n_heads, head_dim))
    ms = np.mean(r * r, axis=-2, keepdims=True)
    return (r / np.sqrt(ms + eps) * np.asarray(w, np.float64)).reshape(x.shape)


def _produce_transposed(feat, wk, wv, k_norm_w, eps, n_head_kv, head_dim):
    x = np.asarray(feat, np.float64)
    k = x @ np.asarray(wk, np.float64)
    v = x @ np.asarray(wv, np.float64)
    return orc.rms_norm_heads(k, k_norm_w, eps, n_head_kv, head_dim), orc.to_f16(v)


def _produce_v_normalised(feat, wk, wv, k_norm_w, eps, n_head_kv, head_dim):
    x = np.asarray(feat, np.float64)
    k = x @ np.asarray(wk, np.float64).T
    v = x @ np.asarray(wv, np.float64).T
    return (orc.rms_norm_heads(k, k_norm_w, eps, n_head_kv, head_dim),
            orc.to_f16(orc.rms_norm_heads(v, k_norm_w, eps, n_head_kv, head_dim)))


def _noise_q_with_k_weight(h, wq, wk, wv, q_norm_w, k_norm_w, eps, n_head, n_head_kv, head_dim):
    x = np.asarray(h, np.float64)
    q = orc.rms_norm_heads(x @ np.asarray(wq, np.float64).T, k_norm_w, eps, n_head, head_dim)
    k, v = orc.produce_rows(h, wk, wv, k_norm_w, eps, n_head_kv, head_dim)
    return q.reshape(x.shape[0], n_head, head_dim), orc.to_f16(k), v


def _noise_q_not_normalised(h, wq, wk, wv, q_norm_w, k_norm_w, eps, n_head, n_head_kv, head_dim):
    x = np.asarray(h, np.float64)
    q = x @ np.asarray(wq, np.float64).T
    k, v = orc.produce_rows(h, wk, wv, k_norm_w, eps, n_head_kv, head_dim)
    return q.reshape(x.shape[0], n_head, head_dim), orc.to_f16(k), v


def _noise_k_not_normalised(h, wq, wk, wv, q_norm_w, k_norm_w, eps, n_head, n_head_kv, head_dim):
    x = np.asarray(h, np.float64)
    q = orc.rms_norm_heads(x @ np.asarray(wq, np.float64).T, q_norm_w, eps, n_head, head_dim)
    k = x @ np.asarray(wk, np.float64).T
    v = orc.to_f16(x @ np.asarray(wv, np.float64).T)
    return q.reshape(x.shape[0], n_head, head_dim), orc.to_f16(k), v


_ORIG_Q8 = orc.q8_0_quantize


def _q8_blocks_of_16(x):
    x = np.asarray(x, np.float64)
    codes = np.empty(x.shape, np.int8)
    scales = []
    for h in range(0, x.shape[-1], 16):
        c, sc = _ORIG_Q8(np.concatenate([x[..., h:h + 16], np.zeros(x.shape[:-1] + (16,))], -1))
        codes[..., h:h + 16] = c[..., :16]
        scales.append(sc[..., 0])
    sc = np.stack(scales, -1)[..., ::2]
    return codes, sc


def _q8_divide_by_128(x):
    x = np.asarray(x, np.float64).astype(np.float32)
    b = x.reshape(x.shape[:-1] + (x.shape[-1] // 32, 32))
    d = (np.max(np.abs(b), -1, keepdims=True) / np.float32(128)).astype(np.float32)
    inv = np.where(d > 0, np.float32(1) / np.where(d > 0, d, 1), 0).astype(np.float32)
    v = (b * inv).astype(np.float64)
    q = np.sign(v) * np.floor(np.abs(v) + 0.5)
    return np.clip(q, -127, 127).astype(np.int8).reshape(x.shape), d[..., 0].astype(np.float16)


def _q8_round_half_even(x):
    x = np.asarray(x, np.float64).astype(np.float32)
    b = x.reshape(x.shape[:-1] + (x.shape[-1] // 32, 32))
    d = (np.max(np.abs(b), -1, keepdims=True) / np.float32(127)).astype(np.float32)
    inv = np.where(d > 0, np.float32(1) / np.where(d > 0, d, 1), 0).astype(np.float32)
    q = np.rint((b * inv).astype(np.float64))
    return np.clip(q, -127, 127).astype(np.int8).reshape(x.shape), d[..., 0].astype(np.float16)


def _q8_dequant_scale_not_rounded(codes, scales):
    c = np.asarray(codes, np.float64)
    b = c.reshape(c.shape[:-1] + (c.shape[-1] // 32, 32))
    s = np.asarray(scales, np.float64) * (1 + 2 ** -9)      # a scale that is not the stored one
    return (b * s[..., None]).reshape(c.shape)


MUTANTS = {
    "q8_0 blocks of 16": ("q8_0_quantize", _q8_blocks_of_16),
    "q8_0 scale max/128": ("q8_0_quantize", _q8_divide_by_128),
    "q8_0 ties to even": ("q8_0_quantize", _q8_round_half_even),
    "q8_0 read-back scale off": ("q8_0_dequantize", _q8_dequant_scale_not_rounded),
    "noise Q takes the k_norm weight": ("project_noise", _noise_q_with_k_weight),
    "noise Q not normalised": ("project_noise", _noise_q_not_normalised),
    "noise K not normalised": ("project_noise", _noise_k_not_normalised),
    "k_norm over the whole row": ("rms_norm_heads", _rms_whole_row),
    "k_norm eps outside the root": ("rms_norm_heads", _rms_eps_outside_root),
    "k_norm weight ignored": ("rms_norm_heads", _rms_weight_ignored),
    "k_norm mean across heads": ("rms_norm_heads", _rms_mean_over_heads),
    "producer weights transposed": ("produce_rows", _produce_transposed),
    "producer normalises V too": ("produce_rows", _produce_v_normalised),
    "slot map off by one": ("slot_of", lambda p, cap: (p + 1) % cap),
    "lo off by one": ("step_window", _step_window_lo_off_by_one),
    "mask_full shows empty slots": ("RingOracle.mask_full", _mask_full_shows_empty_slots),
    "mask_swa ignores swa_window": ("RingOracle.mask_swa", _mask_swa_uses_full_window),
    "mask_swa noise bidirectional": ("RingOracle.mask_swa", _mask_swa_not_causal),
    "rope drops the x2*sin term": ("rope_neox", _rope_drop_term),
    "rope pairs adjacent elements": ("rope_neox", _rope_gptj_pairs),
    "rope exponent -i/d": ("rope_inv_freq", _inv_freq_wrong_exponent),
    "softmax scale 1/d": ("softmax_scale", lambda d: 1.0 / d),
    "kv head h % n_head_kv": ("kv_head_of", lambda h, group: h % 2),
    "f16 by truncation": ("to_f16", _to_f16_truncate),
    "noise keys one position late": ("RingOracle.write_noise", _write_noise_shifted),
    "keys and values swapped": ("masked_attention", _masked_attention_kv_swapped),
    "pad rows not zeroed": ("RingOracle.begin_step", _begin_step_no_pad_zero),
}

PINS = [
    pins.test_geometry_matches_printed_values,
    lambda: [pins.test_tiny_ring_hand_cases(c) for c in pins._golden("tiny_ring.json")["cases"]],
    pins.test_slot_pos_brute_force_and_window_invariant,
    pins.test_mask_counts_closed_form,
    pins.test_empty_context_only_noise_visible,
    pins.test_pad_rows_leave_trash_zero_and_untouched_slots,
    pins.test_f16_round_to_nearest_even,
    pins.test_rope_golden_values,
    pins.test_rope_invariants,
    lambda: pins.test_zero_query_gives_mean_of_visible_positions("full"),
    lambda: pins.test_zero_query_gives_mean_of_visible_positions("swa"),
    pins.test_single_visible_key_returns_its_value,
    pins.test_softmax_scale_is_one_over_sqrt_head_dim,
    pins.test_gqa_head_map,
    pins.test_masked_attention_core_closed_form,
    lambda: pins.test_dense_route_zero_query_closed_form("full"),
    lambda: pins.test_dense_route_zero_query_closed_form("swa"),
    eqv.test_ring_equals_dense_window_tiny_workload,
    pins.test_k_norm_special_cases,
    pins.test_k_norm_epsilon_inside_the_root,
    pins.test_producer_brute_force_small_integers,
    pins.test_producer_permutation_weights_pick_features,
    pins.test_noise_projection_small_integers_and_heads,
    pins.test_noise_projection_query_weight_per_head,
    pins.test_q8_0_hand_values,
    pins.test_q8_0_error_bound_and_brute_force,
]


@contextlib.contextmanager
def _patched(target, repl):
    if "." in target:
        cls_name, attr = target.split(".")
        owner = getattr(orc, cls_name)
    else:
        owner, attr = orc, target
    orig = getattr(owner, attr)
    setattr(owner, attr, repl)
    try:
        yield
    finally:
        setattr(owner, attr, orig)


def test_unmutated_oracle_passes_every_pin():
    for pin in PINS:
        pin()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    target, repl = MUTANTS[name]
    caught = []
    with _patched(target, repl):
        for pin in PINS:
            try:
                pin()
            except (AssertionError, ValueError):
                caught.append(pin)
                break
    assert caught, f"no pin caught the mutant '{name}'"
