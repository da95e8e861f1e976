"""Counter-based seeded generator for K/V rows, queries, noise-block rows, fused features
and the context-row producer's weights.

Every value is a pure function of ``(seed, kind, seq, layer, index, column)``:

* a 32-bit integer finaliser (the xor-shift-multiply "lowbias32" constants published
  in C. Wellons' hash-prospector) mixes the counters into a per-row key and then a
  per-element pair of 32-bit words;
* the four 16-bit halves of those two words are summed (an Irwin-Hall sum of four
  discrete uniforms), centred and scaled to standard deviation ``sigma``.

Only integer operations, one float32 multiply and one float32->float16 rounding are
involved, so a CPU tensor and a CUDA tensor produced here are bit-identical.  That is
what lets the oracle regenerate any context row by absolute position while the GPU
receives the same row.  The functions run on whatever ``device`` they are given.
"""

from __future__ import annotations

import math

import torch

M32 = 0xFFFFFFFF

# Streams of values.  Context rows are keyed by absolute position; queries and
# noise rows by ``step * q_len + i``.
KIND_K_ROW = 1
KIND_V_ROW = 2
KIND_Q = 3
KIND_K_NOISE = 4
KIND_V_NOISE = 5
KIND_FEATURE = 6        # fused target features, keyed by absolute position
KIND_W_K = 7            # producer weights, keyed by output row
KIND_W_V = 8
KIND_K_NORM = 9
KIND_W_Q = 10           # the draft step's query projection
KIND_Q_NORM = 11
KIND_NOISE_H = 12       # noise-block hidden states, keyed by step * q_len + i

# Standard deviation of a sum of four independent uniform integers on [0, 65535].
_IRWIN_HALL4_STD = math.sqrt(4.0 * (65536.0 ** 2 - 1.0) / 12.0)
_IRWIN_HALL4_MEAN = 2 * 65535


def _mul32(x, c: int):
    """``(x * c) mod 2**32`` for values in [0, 2**32) without leaving int64 range."""
    lo = c & 0xFFFF
    hi = c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & M32


def hash32(x):
    """32-bit xor-shift-multiply finaliser; works on Python ints and int64 tensors."""
    x = x & M32
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _stream_key(seed: int, kind: int, seq: int, layer: int) -> int:
    k = hash32((seed & M32) ^ _mul32(kind, 0x9E3779B9))
    k = hash32(k ^ ((seed >> 32) & M32))
    k = hash32(k ^ (seq & M32))
    k = hash32(k ^ (layer & M32))
    return k


def _row_keys(seed: int, kind: int, seq: int, layer: int, index: torch.Tensor) -> torch.Tensor:
    idx = index.to(torch.int64)
    k = _stream_key(seed, kind, seq, layer)
    keys = hash32((idx & M32) ^ k)
    keys = hash32(keys ^ ((idx >> 32) & M32))
    return keys


def gaussian_values(keys: torch.Tensor, width: int, sigma: float) -> torch.Tensor:
    """float32 ``[len(keys), width]``, approximately N(0, sigma^2), bounded by 3.46 sigma."""
    dev = keys.device
    col = torch.arange(width, dtype=torch.int64, device=dev)
    ca = hash32(2 * col + 1)
    cb = hash32(2 * col + 2)
    h1 = hash32(keys[:, None] ^ ca[None, :])
    h2 = hash32(keys[:, None] ^ cb[None, :])
    s = (h1 & 0xFFFF) + (h1 >> 16) + (h2 & 0xFFFF) + (h2 >> 16) - _IRWIN_HALL4_MEAN
    scale = torch.tensor(sigma / _IRWIN_HALL4_STD, dtype=torch.float32, device=dev)
    return s.to(torch.float32) * scale


def _rows(seed, kind, seq, layer, index, width, sigma, chunk_rows=4096):
    index = torch.as_tensor(index, dtype=torch.int64)
    n = index.numel()
    out = torch.empty((n, width), dtype=torch.float32, device=index.device)
    for a in range(0, n, chunk_rows):
        b = min(n, a + chunk_rows)
        out[a:b] = gaussian_values(_row_keys(seed, kind, seq, layer, index[a:b]), width, sigma)
    return out


def context_rows(seed: int, seq: int, layer: int, positions, kv_row: int, sigma: float,
                 device=None, chunk_rows: int = 4096):
    """Pre-RoPE context K and V rows (float16 ``[n, kv_row]``) at absolute ``positions``."""
    pos = torch.as_tensor(positions, dtype=torch.int64, device=device)
    k = _rows(seed, KIND_K_ROW, seq, layer, pos, kv_row, sigma, chunk_rows).to(torch.float16)
    v = _rows(seed, KIND_V_ROW, seq, layer, pos, kv_row, sigma, chunk_rows).to(torch.float16)
    return k, v


def query_block(seed: int, step: int, seq: int, layer: int, q_len: int, n_head: int,
                head_dim: int, sigma: float, device=None):
    """Pre-RoPE noise-block queries, float32 ``[q_len, n_head, head_dim]`` for one step."""
    idx = torch.arange(q_len, dtype=torch.int64, device=device) + step * q_len
    q = _rows(seed, KIND_Q, seq, layer, idx, n_head * head_dim, sigma)
    return q.view(q_len, n_head, head_dim)


def noise_rows(seed: int, step: int, seq: int, layer: int, q_len: int, kv_row: int,
               sigma: float, device=None):
    """Pre-RoPE noise-block K and V rows, float16 ``[q_len, kv_row]`` for one step."""
    idx = torch.arange(q_len, dtype=torch.int64, device=device) + step * q_len
    k = _rows(seed, KIND_K_NOISE, seq, layer, idx, kv_row, sigma).to(torch.float16)
    v = _rows(seed, KIND_V_NOISE, seq, layer, idx, kv_row, sigma).to(torch.float16)
    return k, v


def feature_rows(seed: int, seq: int, positions, hidden: int, sigma: float, device=None,
                 chunk_rows: int = 4096):
    """Fused target features of absolute ``positions``, float16 ``[n, hidden]`` (the same
    vector feeds every layer's producer)."""
    pos = torch.as_tensor(positions, dtype=torch.int64, device=device)
    return _rows(seed, KIND_FEATURE, seq, 0, pos, hidden, sigma, chunk_rows).to(torch.float16)


def producer_weights(seed: int, layer: int, kv_row: int, hidden: int, head_dim: int,
                     device=None):
    """One layer's producer weights: W_k and W_v float16 ``[kv_row, hidden]`` with entries
    of standard deviation 1/sqrt(hidden), and the k_norm weight float32 ``[head_dim]``
    around 1 (standard deviation 0.1)."""
    rows = torch.arange(kv_row, dtype=torch.int64, device=device)
    sig = 1.0 / math.sqrt(hidden)
    wk = _rows(seed, KIND_W_K, 0, layer, rows, hidden, sig).to(torch.float16)
    wv = _rows(seed, KIND_W_V, 0, layer, rows, hidden, sig).to(torch.float16)
    one = torch.zeros(1, dtype=torch.int64, device=device)
    kn = 1.0 + _rows(seed, KIND_K_NORM, 0, layer, one, head_dim, 0.1)[0]
    return wk, wv, kn


def query_weights(seed: int, layer: int, q_rows: int, hidden: int, head_dim: int, device=None):
    """One layer's query projection: W_q float16 ``[q_rows, hidden]`` (standard deviation
    1/sqrt(hidden)) and the q_norm weight float32 ``[head_dim]`` around 1."""
    rows = torch.arange(q_rows, dtype=torch.int64, device=device)
    wq = _rows(seed, KIND_W_Q, 0, layer, rows, hidden, 1.0 / math.sqrt(hidden)).to(torch.float16)
    one = torch.zeros(1, dtype=torch.int64, device=device)
    qn = 1.0 + _rows(seed, KIND_Q_NORM, 0, layer, one, head_dim, 0.1)[0]
    return wq, qn


def noise_hidden(seed: int, step: int, seq: int, layer: int, q_len: int, hidden: int,
                 sigma: float, device=None):
    """Noise-block hidden states of one layer and step, float16 ``[q_len, hidden]``."""
    idx = torch.arange(q_len, dtype=torch.int64, device=device) + step * q_len
    return _rows(seed, KIND_NOISE_H, seq, layer, idx, hidden, sigma).to(torch.float16)
