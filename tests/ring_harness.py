"""Test helper: drives the CUDA ring (through the C ABI binding) and the float64 oracle on
the same seeded workload.  Inputs for the GPU are drawn on the GPU by the seeded
generator; inputs for the oracle are drawn on the CPU by the same generator (the two are
bit-identical, which test_gpu_ring checks).  Nothing here computes ring arithmetic."""

from __future__ import annotations

import numpy as np
import torch

import synth
from oracle import ring_oracle as orc
from speculative_decoding_draft_kv_gb300 import ring as R

# Attention tolerance of the method's parity bar.
ATOL = 2e-3
REL_L2 = 1e-3


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def f16_ulp_diff(a, b) -> np.ndarray:
    """Distance in binary16 units in the last place (+0 and -0 coincide)."""
    def ordered(x):
        u = np.asarray(x, np.float16).view(np.uint16).astype(np.int32)
        mag = u & 0x7FFF
        return np.where(u & 0x8000, -mag, mag)
    return np.abs(ordered(a) - ordered(b))


# K slots: the GPU turns K by RoPE in float32 (angle formed and reduced in float64, then
# float32 sin/cos), the oracle in float64; both round once to F16.  The float32 path is
# off by at most |x1| * |dcos| + |x2| * |dsin| + rounding <= 3e-7 * (|x1| + |x2|) before
# the F16 rounding, and the seeded rows are bounded by 3.46 * 0.5, so a stored K may sit
# one F16 step away, or up to 2e-6 away where the F16 grid is finer than that.
K_ABS = 2e-6


def k_within_tolerance(got, want):
    """(ok, n_not_bit_exact) for F16 K slots against the float64 oracle's F16 K slots."""
    got = np.asarray(got, np.float16)
    want = np.asarray(want, np.float16)
    d = f16_ulp_diff(got, want)
    absdiff = np.abs(got.astype(np.float64) - want.astype(np.float64))
    ok = bool(np.all((d <= 1) | (absdiff <= K_ABS)))
    return ok, int((d > 0).sum())


def f16_spacing(x) -> np.ndarray:
    """Distance between adjacent binary16 values at magnitude |x| (subnormal spacing below
    2^-14)."""
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return np.exp2(e - 10)


def projection_error_bound(feat, w) -> np.ndarray:
    """Bound on |(X W^T) accumulated in float32 - exact|, elementwise.  Each F16 x F16
    product is exact in float32; each of the at most `hidden` additions is off by at most
    one float32 unit (2^-23 relative, so truncating adders are covered) of a partial sum
    no larger than sum |x w|."""
    feat = np.asarray(feat, np.float64)
    w = np.asarray(w, np.float64)
    return feat.shape[-1] * 2.0 ** -23 * (np.abs(feat) @ np.abs(w).T)


def f16_within(got, want_exact, bound) -> bool:
    """F16 values `got` against exact values: |got - exact| <= bound + spacing, i.e. the
    F16 rounding of a value within `bound` of the exact one."""
    got = np.asarray(got, np.float64)
    want_exact = np.asarray(want_exact, np.float64)
    return bool(np.all(np.abs(got - want_exact) <= bound + f16_spacing(np.abs(want_exact) + bound)))


class RowSource:
    """Pre-RoPE context rows by absolute position, drawn on the CPU and cached per
    (seq, layer) as one contiguous window that slides with the requests."""

    def __init__(self, w):
        self.w = w
        self.cache = {}

    def _gen(self, seq, layer, a, b):
        k, v = synth.context_rows(self.w.seed, seq, layer, torch.arange(a, b), self.w.kv_row,
                                  self.w.sigma)
        return k.numpy(), v.numpy()

    def rows(self, seq, layer, pos):
        pos = np.asarray(pos, np.int64)
        if pos.size == 0:
            z = np.zeros((0, self.w.kv_row), np.float16)
            return z, z
        lo, hi = int(pos.min()), int(pos.max()) + 1
        key = (seq, layer)
        if key in self.cache:
            b, k, v = self.cache[key]
            e = b + len(k)
            if lo < b or hi > e:
                ks, vs = [], []
                if lo < b:
                    kk, vv = self._gen(seq, layer, lo, min(b, hi))
                    ks.append(kk), vs.append(vv)
                ov_a, ov_b = max(b, lo), min(e, hi)
                if ov_a < ov_b:
                    ks.append(k[ov_a - b:ov_b - b]), vs.append(v[ov_a - b:ov_b - b])
                if hi > e:
                    kk, vv = self._gen(seq, layer, max(e, lo), hi)
                    ks.append(kk), vs.append(vv)
                k, v, b = np.concatenate(ks), np.concatenate(vs), lo
                self.cache[key] = (b, k, v)
        else:
            k, v = self._gen(seq, layer, lo, hi)
            b = lo
            self.cache[key] = (b, k, v)
        return k[pos - b], v[pos - b]

    def fn(self, seq, layer):
        return lambda pos: self.rows(seq, layer, pos)


class GpuRun:
    """One CUDA ring plus bookkeeping oracles (slot_pos and masks only) per sequence."""

    def __init__(self, w, swa_window=None, tiles_per_split=0, bulk_chunk=0, device="cuda",
                 max_cluster=0, kv_format="f16", step_split=0):
        self.w = w
        self.kv_format = kv_format
        self.swa = w.swa_window if swa_window is None else swa_window
        self.dev = torch.device(device)
        self.ring = R.Ring(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer,
                           w.rope_theta, n_seq=w.n_seq, swa_window=self.swa,
                           bulk_chunk=bulk_chunk, tiles_per_split=tiles_per_split,
                           max_cluster=max_cluster, kv_format=kv_format, step_split=step_split)
        self.g = self.ring.geometry
        # head_dim 2, one head, one layer: only slot_pos and masks are read from these
        self.book = [orc.RingOracle(w.cap, w.q_len, 2, 1, 1, 1, w.rope_theta,
                                    swa_window=self.swa) for _ in range(w.n_seq)]
        self.committed = np.zeros(w.n_seq, np.int64)
        self.rows = RowSource(w)
        self._keep = None

    def close(self):
        self.ring.close()

    def step_rows(self, committed):
        """The new context rows of a step (generated on the device by position), with the
        per-sequence first positions and row offsets the ring takes."""
        w = self.w
        committed = np.asarray(committed, np.int64)
        starts, counts = [], []
        for s in range(w.n_seq):
            st, nn = self.book[s].rows_needed(int(committed[s]))
            assert self.ring.rows_needed(s, int(committed[s])) == (st, nn)
            starts.append(st)
            counts.append(nn)
        n_rows = int(sum(counts))
        row_off = np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int64)
        k_rows = v_rows = None
        if n_rows:
            k_rows = torch.empty((w.n_layer, n_rows, w.kv_row), dtype=torch.float16, device=self.dev)
            v_rows = torch.empty_like(k_rows)
            for s in range(w.n_seq):
                if counts[s] == 0:
                    continue
                pos = torch.arange(starts[s], committed[s], device=self.dev)
                a, b = int(row_off[s]), int(row_off[s]) + counts[s]
                for layer in range(w.n_layer):
                    k, v = synth.context_rows(w.seed, s, layer, pos, w.kv_row, w.sigma, device=self.dev)
                    k_rows[layer, a:b] = k
                    v_rows[layer, a:b] = v
        return committed, np.asarray(starts, np.int64), counts, row_off, k_rows, v_rows

    def _advance_book(self, committed, starts, counts):
        paths = []
        for s in range(self.w.n_seq):
            z = np.zeros((1, counts[s], 2), np.float16)
            paths.append(self.book[s].begin_step(int(committed[s]), z, z, int(starts[s])))
        self.committed = np.asarray(committed, np.int64).copy()
        return paths

    def begin_step(self, committed):
        committed, starts, counts, row_off, k_rows, v_rows = self.step_rows(committed)
        self.ring.begin_step(committed, k_rows, v_rows, row_off, starts)
        self._keep = (k_rows, v_rows)
        return self._advance_book(committed, starts, counts)

    def step(self, committed, kind, q, k_noise, v_noise, o):
        """One whole step through ring_step (begin-step + every layer's attention as one
        replayed CUDA graph); q, k_noise, v_noise, o: per-layer device tensors."""
        committed, starts, counts, row_off, k_rows, v_rows = self.step_rows(committed)
        self.ring.step(committed, k_rows, v_rows, row_off, starts, kind, q, k_noise, v_noise, o)
        self._keep = (k_rows, v_rows)
        return self._advance_book(committed, starts, counts)

    def inputs(self, step, layer, device):
        w = self.w
        qs, ks, vs = [], [], []
        for s in range(w.n_seq):
            qs.append(synth.query_block(w.seed, step, s, layer, w.q_len, w.n_head, w.head_dim,
                                        w.sigma, device=device))
            k, v = synth.noise_rows(w.seed, step, s, layer, w.q_len, w.kv_row, w.sigma, device=device)
            ks.append(k)
            vs.append(v)
        return torch.stack(qs), torch.stack(ks), torch.stack(vs)

    def attend(self, step, layer, kind):
        q, kn, vn = self.inputs(step, layer, self.dev)
        o = torch.empty_like(q)
        self.ring.attend(layer, kind, q, kn, vn, o)
        torch.cuda.synchronize()
        return o.cpu().numpy()

    def expected(self, step, layer, kind, seq, heads=None):
        w = self.w
        q = synth.query_block(w.seed, step, seq, layer, w.q_len, w.n_head, w.head_dim, w.sigma)
        kn, vn = synth.noise_rows(w.seed, step, seq, layer, w.q_len, w.kv_row, w.sigma)
        return orc.attend_dense(int(self.committed[seq]), w.cap, self.rows.fn(seq, layer),
                                q.numpy(), kn.numpy(), vn.numpy(), w.head_dim, w.n_head_kv,
                                w.n_head, w.rope_theta, kind=kind, swa_window=self.swa,
                                heads=heads, kv_format=self.kv_format)

    def check_slots_and_masks(self, seqs=None):
        for s in (range(self.w.n_seq) if seqs is None else seqs):
            b = self.book[s]
            np.testing.assert_array_equal(self.ring.slot_pos(s), b.slot_pos.astype(np.int32))
            kinds = ["full"] + (["swa"] if self.swa else [])
            for kind in kinds:
                want = b.mask(kind)
                got = self.ring.mask(s, kind)
                assert got.view(np.uint32).tobytes() == want.view(np.uint32).tobytes(), (s, kind)
                np.testing.assert_array_equal(self.ring.tile_flags(s, kind),
                                              expected_tile_flags(want, self.g["tile_slots"]))

    def check_kv_slots(self, seq, layer, slots):
        """Sampled slots of K/V against RoPE'd rows regenerated by position."""
        w = self.w
        k, v = self.ring.kv(seq, layer)
        sp = self.book[seq].slot_pos
        slots = [s for s in slots if sp[s] >= 0]
        pos = np.array([sp[s] for s in slots], np.int64)
        if not len(pos):
            return 0
        kr, vr = self.rows.rows(seq, layer, pos)
        want_k = orc.to_f16(orc.rope_rows(kr.astype(np.float64), pos, w.n_head_kv, w.head_dim,
                                          w.rope_theta))
        np.testing.assert_array_equal(v[slots], vr)
        ok, inexact = k_within_tolerance(k[slots], want_k)
        assert ok and inexact <= 0.01 * want_k.size, inexact
        assert np.all(k[self.g["trash_slot"]] == 0) and np.all(v[self.g["trash_slot"]] == 0)
        return inexact


    def check_kv_slots_q8(self, seq, layer, slots):
        """q8_0 rings: sampled slots' codes and scales against the oracle's quantisation of
        the rows regenerated by position (V exact; K within q8_k_within)."""
        w = self.w
        kc, ks, vc, vs = self.ring.kv_q8(seq, layer)
        sp = self.book[seq].slot_pos
        slots = [s for s in slots if sp[s] >= 0]
        pos = np.array([sp[s] for s in slots], np.int64)
        t = self.g["trash_slot"]
        assert not kc[t].any() and not vc[t].any()
        assert not ks[t].view(np.uint16).any() and not vs[t].view(np.uint16).any()
        if not len(pos):
            return 0
        kr, vr = self.rows.rows(seq, layer, pos)
        wkc, wks = orc.q8_0_quantize(orc.rope_rows(kr.astype(np.float64), pos, w.n_head_kv,
                                                   w.head_dim, w.rope_theta))
        wvc, wvs = orc.q8_0_quantize(vr)
        np.testing.assert_array_equal(vc[slots], wvc)
        np.testing.assert_array_equal(vs[slots].view(np.uint16), wvs.view(np.uint16))
        return q8_k_within(kc[slots], ks[slots], wkc, wks)


def q8_k_within(kc, ks, want_kc, want_ks, frac=0.01):
    """K codes and scales of a q8_0 ring against the oracle's.  The GPU rotates in float32
    with CUDA's sin/cos and the oracle in float64, so a rotated value can differ in its
    last float32 bits: a block maximum, and so its scale, may move by one F16 ulp and a
    code sitting on a rounding boundary by one.  Returns the number of differing codes
    (at most `frac` of all)."""
    dc = np.abs(kc.astype(np.int32) - want_kc.astype(np.int32))
    assert dc.max(initial=0) <= 1, int(dc.max())
    assert f16_ulp_diff(ks, want_ks).max(initial=0) <= 1
    n = int((dc != 0).sum())
    assert n <= frac * kc.size, (n, kc.size)
    return n


def expected_tile_flags(mask, tile):
    """0: no slot of the tile visible to any row; 1: every slot of a full-size tile
    visible to every row; 2: anything else."""
    q_len, kv_total = mask.shape
    n_tiles = (kv_total + tile - 1) // tile
    out = np.zeros(n_tiles, np.uint8)
    for t in range(n_tiles):
        seg = mask[:, t * tile:(t + 1) * tile] == 0
        if not seg.any():
            out[t] = 0
        elif seg.shape[1] == tile and seg.all():
            out[t] = 1
        else:
            out[t] = 2
    return out


def assert_close(got, want, what=""):
    err = float(np.abs(got - want).max())
    rl2 = rel_l2(got, want)
    assert err <= ATOL and rl2 <= REL_L2, f"{what}: max abs {err:.3g}, rel L2 {rl2:.3g}"
    return err, rl2
