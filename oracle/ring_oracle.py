"""Float64 CPU oracle of the DFlash draft-KV ring step.

TEST INFRASTRUCTURE.  This module states, plainly and slowly, what the ring step
computes.  Only ``tests/``, the smoke check in ``__graft_entry__`` and the CPU-baseline
and reference legs of ``bench.py`` may import it.  It shares no code with the CUDA
path, never loads the CUDA library, and the product path never imports it.

Source: the page "DFLASH2_RING_PORT.md" (DFlash2 draft KV-ring port to llama.cpp):
  * section 1.1 -- geometry fixed by draft_kv_init;
  * section 1.2 -- mod-cap slot map: slot = p % cap, slot_pos[slot] = p;
  * section 1.3 -- begin_step window arithmetic, fold-in vs bulk append, noise positions;
  * section 1.4 -- mask_full and mask_swa;
  * section 1.7 -- the ring equals a recompute of the full window; F16 memory formula;
  * section 2.2 -- the naive seq_rm roll (used only as a negative model).

Readings taken where the page is silent (each is listed in the design notes):
  R1  trash_slot and the alignment pad slots [cap+q_len+1, kv_total) are masked -inf;
  R2  pad rows of a fold-in step are written as zeros to trash_slot;
  R3  slot_pos starts at -1 (an empty slot is never inside a window, since lo >= 0);
  R4  softmax scale is 1/sqrt(head_dim);
  R5  RoPE is the NeoX form over the whole head: pair (i, i + d/2) turns by
      p * theta^(-2i/d);
  R6  RoPE is applied to context K at its position p, to noise K at committed + j and
      to the queries at committed + i; V is never rotated;
  R7  query head h reads kv head h // (n_head / n_head_kv);
  R8  K/V live in F16 (round to nearest even after a float64 rotation); Q and O are
      real-valued (float64 here);
  R9  under mask_swa, noise slot cap+j is visible to query row i iff j <= i, and the
      context window is anchored at committed for every row;
  R10 rows handed to begin_step cover [first_pos, committed); only [start, committed)
      is stored, positions below lo are ignored.

The context-row producer (page "DFLASH2_RING_PORT.md", test 11, point 4 of the refuted
hypotheses: the draft's context K/V come from a shallow injection of the fused target
features, wk/wv times the features, then k_norm, then RoPE):
  P1  the pre-RoPE context row of position p is K = k_norm(W_k x_p), V = W_v x_p, with
      x_p the fused feature vector of p (F16, width ``hidden``, shared by the layers)
      and W_k, W_v F16 [kv_row, hidden] per layer;
  P2  k_norm is an RMS norm over each kv head's head_dim slice,
      y = x / sqrt(mean(x^2) + eps) * w, with one learned weight w [head_dim] per layer
      shared by the heads and eps = 1e-6;
  P3  K then takes RoPE at p (R5, R6) and is rounded to F16; V is rounded to F16
      straight from the product.

The whole draft step (the page's one-graph draft forward, section 1.5, with the noise
block fed in per layer, section 1.6):
  F1  a layer's noise-block rows come from its input hidden states h (one row per noise
      position): Q = q_norm(W_q h), K = k_norm(W_k h), V = W_v h, with the same W_k, W_v
      and k_norm as the context rows and q_norm an RMS norm over each query head with its
      own weight [head_dim] (P2's form); K and V are handed to the attention as F16
      pre-RoPE rows, Q as real pre-RoPE values;
  F2  each layer attends with its own mask kind (full or SWA), a fixed per-layer pattern.

The quantised ring (the port's ~48 MiB draft-KV figure, section 1.7, is consistent with a
q8_0 cache):
  Q1  q8_0 blocks are 32 consecutive values of one head's row (head_dim / 32 blocks per
      head); scale d = max|x| / 127 and codes round(x / d), rounding half away from zero,
      computed in float32 (x * (1/d)); d is stored as F16 and a value reads back as
      code * d_f16; an all-zero block has d = 0 and codes 0;
  Q2  K is quantised straight from its rotated value (no F16 rounding first), V from its
      input value; noise rows like context rows; pad rows are all-zero blocks.

Precision: float64 throughout, except for the F16 storage of K and V that the page
fixes.  Parity pins for every function here live in tests/test_oracle_*.py.
"""

from __future__ import annotations

import math

import numpy as np

NEG_INF = np.float32(-np.inf)


# ---------------------------------------------------------------------------
# section 1.1: geometry
# ---------------------------------------------------------------------------

def align_up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


def geometry(cap: int, q_len: int, head_dim: int, n_head_kv: int, n_layer: int) -> dict:
    """Ring geometry (section 1.1) and the F16 cache size (section 1.7)."""
    a_step = 2 * q_len + 2
    trash_slot = cap + q_len
    kv_total = align_up(cap + q_len + 1, 32)
    kv_row = head_dim * n_head_kv
    cache_bytes = 2 * n_layer * kv_row * kv_total * 2   # K and V, 2 bytes per F16
    return dict(cap=cap, q_len=q_len, a_step=a_step, trash_slot=trash_slot,
                kv_total=kv_total, kv_row=kv_row, n_layer=n_layer,
                cache_bytes=cache_bytes)


# ---------------------------------------------------------------------------
# section 1.3: window arithmetic of begin_step
# ---------------------------------------------------------------------------

def step_window(committed: int, next_pos: int, cap: int) -> tuple[int, int, int, int]:
    """(win, lo, start, n_new) of one begin_step."""
    win = min(committed, cap)
    lo = committed - win
    start = max(next_pos, lo)
    n_new = committed - start
    return win, lo, start, n_new


def slot_of(p: int, cap: int) -> int:
    """Section 1.2: the slot of absolute position p is p mod cap."""
    return p % cap


def kv_head_of(h: int, group: int) -> int:
    """Reading R7: query head h reads kv head h // group (group = n_head / n_head_kv)."""
    return h // group


def softmax_scale(head_dim: int) -> float:
    """Reading R4."""
    return 1.0 / math.sqrt(head_dim)


def swa_low(committed: int, cap: int, swa_window: int) -> int:
    """Lower bound of the SWA window (section 1.4): committed - min(swa_window, win)."""
    win = min(committed, cap)
    eff_win = min(swa_window, win)
    return committed - eff_win


# ---------------------------------------------------------------------------
# storage rounding and RoPE
# ---------------------------------------------------------------------------

def to_f16(x) -> np.ndarray:
    """Round float64 values to IEEE binary16, nearest-even (numpy's direct conversion)."""
    return np.asarray(x, dtype=np.float64).astype(np.float16)


Q8_BLOCK = 32


def q8_0_quantize(x):
    """Codes (int8, same shape) and F16 scales (one per 32 values along the last axis) of
    ``x`` (Q1).  The decisions are taken in float32."""
    x = np.asarray(x, dtype=np.float64).astype(np.float32)
    shp = x.shape
    b = x.reshape(shp[:-1] + (shp[-1] // Q8_BLOCK, Q8_BLOCK))
    amax = np.max(np.abs(b), axis=-1, keepdims=True)
    d = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(d > 0, np.float32(1.0) / np.where(d > 0, d, np.float32(1.0)),
                       np.float32(0.0)).astype(np.float32)
    v = (b * inv).astype(np.float32).astype(np.float64)
    q = np.sign(v) * np.floor(np.abs(v) + 0.5)               # half away from zero
    codes = np.clip(q, -127, 127).astype(np.int8).reshape(shp)
    return codes, d[..., 0].astype(np.float16)


def q8_0_dequantize(codes, scales) -> np.ndarray:
    """float64 values of q8_0 ``codes`` with F16 ``scales`` (one per 32 codes)."""
    c = np.asarray(codes, dtype=np.float64)
    shp = c.shape
    b = c.reshape(shp[:-1] + (shp[-1] // Q8_BLOCK, Q8_BLOCK))
    return (b * np.asarray(scales, dtype=np.float64)[..., None]).reshape(shp)


def q8_0_round_trip(x) -> np.ndarray:
    return q8_0_dequantize(*q8_0_quantize(x))


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * i / head_dim)


def rope_neox(x, pos, theta: float) -> np.ndarray:
    """Rotate the last axis (one head) at absolute position(s) ``pos`` (reading R5).

    ``x``: [..., head_dim]; ``pos`` broadcasts against ``x.shape[:-1]``.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def rope_rows(rows, pos, n_heads: int, head_dim: int, theta: float) -> np.ndarray:
    """RoPE of rows laid out [..., n_heads * head_dim] (head-major), float64 result."""
    rows = np.asarray(rows, dtype=np.float64)
    shp = rows.shape
    r = rows.reshape(shp[:-1] + (n_heads, head_dim))
    p = np.asarray(pos, dtype=np.float64)[..., None]        # same angle for every head
    return rope_neox(r, p, theta).reshape(shp)


# ---------------------------------------------------------------------------
# context-row producer (P1-P3): projection, per-head RMS norm
# ---------------------------------------------------------------------------

def rms_norm_heads(x, w, eps: float, n_heads: int, head_dim: int) -> np.ndarray:
    """RMS norm of every head slice of rows [..., n_heads * head_dim] (P2), float64.

    Each head's slice is divided by the root of its mean square plus ``eps`` and then
    multiplied elementwise by ``w`` [head_dim].
    """
    x = np.asarray(x, dtype=np.float64)
    shp = x.shape
    r = x.reshape(shp[:-1] + (n_heads, head_dim))
    ms = np.mean(r * r, axis=-1, keepdims=True)
    y = r / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)
    return y.reshape(shp)


def produce_rows(feat, wk, wv, k_norm_w, eps: float, n_head_kv: int, head_dim: int):
    """Context rows of fused features ``feat`` [n, hidden] for one layer (P1, P2).

    Returns the pre-RoPE K rows (float64, not rounded: RoPE and the F16 rounding follow,
    P3) and the V rows (F16), both [n, n_head_kv * head_dim].
    """
    x = np.asarray(feat, dtype=np.float64)
    k = x @ np.asarray(wk, dtype=np.float64).T
    v = x @ np.asarray(wv, dtype=np.float64).T
    return rms_norm_heads(k, k_norm_w, eps, n_head_kv, head_dim), to_f16(v)


def project_noise(h, wq, wk, wv, q_norm_w, k_norm_w, eps: float, n_head: int, n_head_kv: int,
                  head_dim: int):
    """Noise-block rows of one layer from its hidden states ``h`` [q_len, hidden] (F1).

    Returns Q (float64 [q_len, n_head, head_dim], pre-RoPE), K and V (F16
    [q_len, n_head_kv * head_dim], pre-RoPE), as the attention takes them.
    """
    x = np.asarray(h, dtype=np.float64)
    q = rms_norm_heads(x @ np.asarray(wq, dtype=np.float64).T, q_norm_w, eps, n_head, head_dim)
    k, v = produce_rows(h, wk, wv, k_norm_w, eps, n_head_kv, head_dim)
    return q.reshape(x.shape[0], n_head, head_dim), to_f16(k), v


# ---------------------------------------------------------------------------
# attention core: softmax(scale * q.k + mask) . v, float64
# ---------------------------------------------------------------------------

def masked_attention(q, k, v, mask, scale: float) -> np.ndarray:
    """O[r] = sum_s softmax_s(scale * q[r].k[s] + mask[r, s]) v[s].

    q [R, d], k [N, d], v [N, d], mask [R, N] holding 0 or -inf.  Every row must see at
    least one key.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    s = (q @ k.T) * scale + np.asarray(mask, np.float64)
    m = s.max(axis=1, keepdims=True)
    if not np.all(np.isfinite(m)):
        raise ValueError("a query row sees no key")
    w = np.exp(s - m)
    w = w / w.sum(axis=1, keepdims=True)
    return w @ v


# ---------------------------------------------------------------------------
# O1: the ring state, step by step (sections 1.1-1.4)
# ---------------------------------------------------------------------------

class RingOracle:
    """One sequence's draft-KV ring: slot_pos, F16 K/V tensors and the masks."""

    def __init__(self, cap, q_len, head_dim, n_head_kv, n_head, n_layer, rope_theta,
                 swa_window=0, bulk_chunk=1024, kv_format="f16"):
        if n_head % n_head_kv:
            raise ValueError("n_head must be a multiple of n_head_kv")
        g = geometry(cap, q_len, head_dim, n_head_kv, n_layer)
        self.cap, self.q_len = cap, q_len
        self.head_dim, self.n_head_kv, self.n_head = head_dim, n_head_kv, n_head
        self.n_layer, self.theta = n_layer, float(rope_theta)
        self.swa_window, self.bulk_chunk = swa_window, bulk_chunk
        self.a_step, self.trash_slot = g["a_step"], g["trash_slot"]
        self.kv_total, self.kv_row = g["kv_total"], g["kv_row"]
        # section 1.1: separate F16 tensors, zeroed once; one row of kv_row per slot
        self.kv_format = kv_format
        if kv_format == "q8_0":
            # codes and F16 scales (Q1); self.k / self.v hold what the slots read back as
            nb = self.kv_row // Q8_BLOCK
            self.kq = np.zeros((n_layer, self.kv_total, self.kv_row), np.int8)
            self.vq = np.zeros((n_layer, self.kv_total, self.kv_row), np.int8)
            self.ks = np.zeros((n_layer, self.kv_total, nb), np.float16)
            self.vs = np.zeros((n_layer, self.kv_total, nb), np.float16)
            self.k = np.zeros((n_layer, self.kv_total, self.kv_row), np.float64)
            self.v = np.zeros((n_layer, self.kv_total, self.kv_row), np.float64)
        else:
            self.k = np.zeros((n_layer, self.kv_total, self.kv_row), np.float16)
            self.v = np.zeros((n_layer, self.kv_total, self.kv_row), np.float16)
        self.slot_pos = np.full(cap, -1, np.int64)      # reading R3
        self.next_pos = 0
        self.committed = None
        self.last_path = None

    # -- section 1.3 ------------------------------------------------------
    def rows_needed(self, committed: int) -> tuple[int, int]:
        _, _, start, n_new = step_window(committed, self.next_pos, self.cap)
        return start, n_new

    def _put(self, layer: int, slot: int, k_rot, v_row) -> None:
        """Store a rotated K row and a V row in one slot: F16, or q8_0 blocks (Q1, Q2)."""
        if self.kv_format == "q8_0":
            self.kq[layer, slot], self.ks[layer, slot] = q8_0_quantize(k_rot)
            self.vq[layer, slot], self.vs[layer, slot] = q8_0_quantize(v_row)
            self.k[layer, slot] = q8_0_dequantize(self.kq[layer, slot], self.ks[layer, slot])
            self.v[layer, slot] = q8_0_dequantize(self.vq[layer, slot], self.vs[layer, slot])
        else:
            self.k[layer, slot] = to_f16(k_rot)
            self.v[layer, slot] = v_row

    def _store(self, p: int, k_row, v_row) -> None:
        """Section 1.2: the row of absolute position p goes to slot p % cap."""
        slot = slot_of(p, self.cap)
        for layer in range(self.n_layer):
            kr = rope_rows(k_row[layer], p, self.n_head_kv, self.head_dim, self.theta)
            self._put(layer, slot, kr, v_row[layer])
        self.slot_pos[slot] = p

    def begin_step(self, committed: int, k_rows, v_rows, first_pos: int) -> str:
        """Append the rows of [start, committed); rebuilds nothing else.

        ``k_rows``/``v_rows``: F16 [n_layer, n, kv_row] for positions first_pos + r.
        Returns the path taken: "bulk" or "fold".
        """
        if committed < self.next_pos:
            raise ValueError("committed went backwards")
        win, lo, start, n_new = step_window(committed, self.next_pos, self.cap)
        if n_new > 0:
            n_rows = np.asarray(k_rows).shape[1]
            if first_pos > start or first_pos + n_rows < committed:
                raise ValueError("rows do not cover [start, committed)")
        if n_new > self.a_step:
            # draft_kv_bulk_append: chunks of bulk_chunk rows, every row to its slot
            for c0 in range(start, committed, self.bulk_chunk):
                for p in range(c0, min(committed, c0 + self.bulk_chunk)):
                    r = p - first_pos
                    self._store(p, k_rows[:, r], v_rows[:, r])
            path = "bulk"
        else:
            # fold-in: a_step rows, the real ones first, pad rows to trash_slot (R2)
            for i in range(self.a_step):
                if i < n_new:
                    p = start + i
                    r = p - first_pos
                    self._store(p, k_rows[:, r], v_rows[:, r])
                else:
                    self.k[:, self.trash_slot] = 0
                    self.v[:, self.trash_slot] = 0
                    if self.kv_format == "q8_0":
                        self.kq[:, self.trash_slot] = 0
                        self.vq[:, self.trash_slot] = 0
                        self.ks[:, self.trash_slot] = 0
                        self.vs[:, self.trash_slot] = 0
            path = "fold"
        self.next_pos = committed
        self.committed = committed
        self.last_path = path
        return path

    # -- section 1.4 ------------------------------------------------------
    def mask_full(self) -> np.ndarray:
        """[q_len, kv_total] float32: 0 where visible, -inf elsewhere."""
        c = self.committed
        win = min(c, self.cap)
        lo = c - win
        m = np.full((self.q_len, self.kv_total), NEG_INF, np.float32)
        for s in range(self.cap):
            p = self.slot_pos[s]
            if lo <= p < c:
                m[:, s] = 0.0
        m[:, self.cap:self.cap + self.q_len] = 0.0       # noise block, bidirectional
        return m

    def mask_swa(self) -> np.ndarray:
        """[q_len, kv_total] float32, SWA window anchored at committed; causal noise (R9)."""
        c = self.committed
        slo = swa_low(c, self.cap, self.swa_window)
        m = np.full((self.q_len, self.kv_total), NEG_INF, np.float32)
        for s in range(self.cap):
            p = self.slot_pos[s]
            if slo <= p < c:
                m[:, s] = 0.0
        for i in range(self.q_len):
            for j in range(self.q_len):
                if j <= i:
                    m[i, self.cap + j] = 0.0
        return m

    def mask(self, kind: str) -> np.ndarray:
        return self.mask_full() if kind == "full" else self.mask_swa()

    # -- noise block and masked attention over the kv_total slots -----------
    def write_noise(self, layer: int, k_noise, v_noise) -> None:
        """Noise rows j go to slots cap + j with RoPE at committed + j (section 1.3)."""
        c = self.committed
        for j in range(self.q_len):
            kr = rope_rows(k_noise[j], c + j, self.n_head_kv, self.head_dim, self.theta)
            self._put(layer, self.cap + j, kr, v_noise[j])

    def attend(self, layer: int, q, k_noise, v_noise, kind: str = "full") -> np.ndarray:
        """O [q_len, n_head, head_dim] float64 of the noise queries over the ring."""
        self.write_noise(layer, k_noise, v_noise)
        c = self.committed
        G = self.n_head // self.n_head_kv
        d = self.head_dim
        pos_q = c + np.arange(self.q_len)
        qr = rope_neox(np.asarray(q, np.float64), pos_q[:, None], self.theta)   # [q, H, d]
        mask = self.mask(kind)
        kf = self.k[layer].astype(np.float64).reshape(self.kv_total, self.n_head_kv, d)
        vf = self.v[layer].astype(np.float64).reshape(self.kv_total, self.n_head_kv, d)
        out = np.zeros((self.q_len, self.n_head, d), np.float64)
        for h in range(self.n_head):
            g = kv_head_of(h, G)
            out[:, h, :] = masked_attention(qr[:, h, :], kf[:, g, :], vf[:, g, :], mask,
                                            softmax_scale(d))
        return out


# ---------------------------------------------------------------------------
# O2: dense attention over exactly the window (section 1.7), no ring at all
# ---------------------------------------------------------------------------

def attend_dense(committed, cap, rows_fn, q, k_noise, v_noise, head_dim, n_head_kv, n_head,
                 rope_theta, kind="full", swa_window=0, heads=None, kv_format="f16") -> np.ndarray:
    """Attention of the q_len noise queries over the positions [lo, committed) plus the
    noise block, computed from the rows themselves.

    ``rows_fn(positions) -> (k, v)`` returns the pre-RoPE F16 context rows
    [len(positions), n_head_kv * head_dim] of the layer in question.  Under ``kind="swa"``
    the window is [committed - min(swa_window, win), committed) and the noise block is
    causal.  ``heads`` restricts the output to a subset of query heads (others are 0).
    """
    c = int(committed)
    q = np.asarray(q, np.float64)
    q_len = q.shape[0]
    win = min(c, cap)
    lo = c - win
    if kind == "swa":
        lo = c - min(swa_window, win)
    pos = np.arange(lo, c, dtype=np.int64)
    kc, vc = rows_fn(pos)
    # the stored form of every key and value: F16, or q8_0 blocks read back (Q1, Q2)
    store = q8_0_round_trip if kv_format == "q8_0" else to_f16
    kc = store(rope_rows(np.asarray(kc, np.float64), pos, n_head_kv, head_dim, rope_theta))
    jn = np.arange(q_len)
    kn = store(rope_rows(np.asarray(k_noise, np.float64), c + jn, n_head_kv, head_dim,
                         rope_theta))
    keys = np.concatenate([kc, kn], axis=0).astype(np.float64)
    vals = np.concatenate([np.asarray(store(vc), np.float64), np.asarray(store(v_noise), np.float64)],
                          axis=0)
    n_ctx = len(pos)
    mask = np.zeros((q_len, n_ctx + q_len), np.float64)
    if kind == "swa":
        for i in range(q_len):
            for j in range(q_len):
                if j > i:
                    mask[i, n_ctx + j] = -np.inf
    qr = rope_neox(q, (c + np.arange(q_len))[:, None], rope_theta)
    G = n_head // n_head_kv
    keys = keys.reshape(-1, n_head_kv, head_dim)
    vals = vals.reshape(-1, n_head_kv, head_dim)
    out = np.zeros((q_len, n_head, head_dim), np.float64)
    for h in (range(n_head) if heads is None else heads):
        g = kv_head_of(h, G)
        out[:, h, :] = masked_attention(qr[:, h, :], keys[:, g, :], vals[:, g, :], mask,
                                        softmax_scale(head_dim))
    return out


# ---------------------------------------------------------------------------
# section 2.2: the naive roll (negative model, never the reference)
# ---------------------------------------------------------------------------

class NaiveRollOracle:
    """The broken scheme of section 2.2: a plain cache of ``n_ctx`` cells filled in
    arrival order, oldest cells evicted when full, the noise block taking cells too, and
    attention over every resident cell with no window mask.  Used only to show that the
    parity checks can tell it apart from the ring once evictions begin."""

    def __init__(self, n_ctx, q_len, head_dim, n_head_kv, n_head, rope_theta):
        self.n_ctx, self.q_len = n_ctx, q_len
        self.head_dim, self.n_head_kv, self.n_head = head_dim, n_head_kv, n_head
        self.theta = float(rope_theta)
        self.cells = []          # (pos, k_row_f16_roped, v_row_f16)
        self.next_pos = 0
        self.committed = 0

    def _push(self, pos, k, v):
        if len(self.cells) == self.n_ctx:
            self.cells.pop(0)
        self.cells.append((pos, k, v))

    def begin_step(self, committed, k_rows, v_rows, first_pos):
        for p in range(self.next_pos, committed):
            r = p - first_pos
            if r < 0:
                continue
            k = to_f16(rope_rows(k_rows[r], p, self.n_head_kv, self.head_dim, self.theta))
            self._push(p, k, np.asarray(v_rows[r]))
        self.next_pos = committed
        self.committed = committed

    def attend(self, q, k_noise, v_noise):
        c = self.committed
        for j in range(self.q_len):
            k = to_f16(rope_rows(k_noise[j], c + j, self.n_head_kv, self.head_dim, self.theta))
            self._push(c + j, k, np.asarray(v_noise[j]))
        keys = np.stack([cell[1] for cell in self.cells]).astype(np.float64)
        vals = np.stack([cell[2] for cell in self.cells]).astype(np.float64)
        # the noise cells are popped again after the step, as a decode batch would be
        self.cells = self.cells[:-self.q_len]
        keys = keys.reshape(-1, self.n_head_kv, self.head_dim)
        vals = vals.reshape(-1, self.n_head_kv, self.head_dim)
        qr = rope_neox(np.asarray(q, np.float64), (c + np.arange(self.q_len))[:, None],
                       self.theta)
        G = self.n_head // self.n_head_kv
        out = np.zeros((self.q_len, self.n_head, self.head_dim))
        mask = np.zeros((self.q_len, keys.shape[0]))
        for h in range(self.n_head):
            g = kv_head_of(h, G)
            out[:, h, :] = masked_attention(qr[:, h, :], keys[:, g, :], vals[:, g, :], mask,
                                            softmax_scale(self.head_dim))
        return out
