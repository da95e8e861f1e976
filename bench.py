"""Benchmark of the DFlash draft-KV ring step on GB300 (one JSON line on stdout).

A step is one ring_begin_step for every sequence plus one ring_attend per layer, all
through the C ABI, on a synthetic workload (seeded inputs; no model weights exist for
this path).  Default workload: one sequence, five layers, cap 4096, q_len 8, prefilled
to 8192 committed tokens and then advanced by the page's acceptance histogram.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--workload 2|3|4|5] [--mask full|swa] [--step-split S]

The line also carries, under "configs", the method's other roofline workloads measured
the same way (cap 32768 x 16 sequences; cap 4096 x 64 sequences with mask_full and with
mask_swa, window 2048), each with its own roofline, oracle baseline and state check.

Under torchrun every rank runs its own independent rings (weak scaling, no collective on
the data path); rank 0 prints the line with the max-over-ranks time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ring attention steps/s and HBM GB/s (% of GB300 peak) at cap 4096, q_len 8"
UNIT = "steps/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the split-KV attention kernel,
# from one ncu capture, keyed by workload; valid only for the kernel code it was taken on
# (kernel = _code_hash of attn_kernels.cu: sha256[:16] without comments and whitespace).
NCU_TRAFFIC = {
    "steady_decode_cap4096_s1_l5": {"bytes": 33_856_128, "kernel": "2ee0f6a3f6510f19",
                                    "source": "profiles/attend_cluster_steady_decode_cap4096_s1_l5.md"},
    # captured on 4 of the 16 sequences (538,202,368 B read + 14,991,872 B written per
    # launch) and scaled by the sequences a launch processes: every sequence's visible rows
    # are read once, so the traffic grows in proportion
    "large_ring_cap32768_s16_l5": {"bytes": 4 * (538_202_368 + 14_991_872), "kernel": "2ee0f6a3f6510f19",
                                   "source": "profiles/attend_plain_large_cap32768_s4_l5.md"},
}
# dram__bytes_read.sum + dram__bytes_write.sum per launch of the producer kernels, keyed as
# above (kernel = _code_hash of produce_kernels.cu or produce_tc.cu)
PRODUCE_TRAFFIC = {
    "steady_decode_cap4096_s1_l5": {"bytes": 84_903_552, "kernel": "1117b6f1d0ffc179",
                                    "source": "profiles/produce_steady_decode_cap4096_s1_l5.md"},
    # the tensor-core kernel (produce_tc.cu) on the legacy recompute's 4096 rows
    "steady_decode_cap4096_s1_l5_legacy": {"bytes": 181_065_984, "kernel": "c446e1838298dba4",
                                           "source": "profiles/produce_tc_legacy_recompute_cap4096_s1_l5.md"},
}


def _code_hash(text: str) -> str:
    """sha256[:16] of a CUDA source's code: comments and whitespace removed, so that a
    change to the comments alone leaves a capture of the kernel valid."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()[:16]


def _kernel_source_hash(name: str = "attn_kernels.cu") -> str:
    p = os.path.join(ROOT, "speculative_decoding_draft_kv_gb300", "csrc", name)
    with open(p) as f:
        return _code_hash(f.read())


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _tensor_peak():
    """(bf16 dense TFLOP/s, source): MEASURED_PEAKS.json's burst figure, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def _dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms while running."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.path = None
        self.gpu_id = gpu_id

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS),
                   "--format=csv,noheader,nounits", "-lms", "200"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        # nvidia-smi's own start-up (driver and NVML initialisation) must not fall inside
        # the timed region: wait for its first sample
        t_end = time.time() + 5.0
        while time.time() < t_end and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == len(self.FIELDS):
                    rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[4 + k] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------------------
# workload preparation (inputs resident in HBM before timing)
# ----------------------------------------------------------------------------------------

class Prepared:
    pass


def prepare(w, n_steps, rank, dev):
    """Everything the timed steps read, resident in HBM: one buffer with every step's new
    context rows (a step addresses its rows through row_off), fixed per-layer query,
    noise-row and output buffers."""
    import numpy as np
    import torch

    import synth

    # row 0 is the untimed first call (the prefill where the workload has one)
    sched = synth.commit_schedule(w, n_steps + (0 if w.kind in ("decode", "batched", "large") else 1))
    P = Prepared()
    P.sched = sched
    S, L = w.n_seq, w.n_layer
    seq_ids = [rank * S + s for s in range(S)]
    next_pos = np.zeros(S, np.int64)
    plan = []
    total = 0
    for t in range(sched.shape[0]):
        c = sched[t]
        start = np.maximum(next_pos, c - np.minimum(c, w.cap))
        counts = (c - start).astype(np.int64)
        row_off = total + np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int64)
        plan.append((c.copy(), row_off, start.copy(), counts))
        total += int(counts.sum())
        next_pos = c.copy()
    P.k_all = torch.empty((L, max(total, 1), w.kv_row), dtype=torch.float16, device=dev)
    P.v_all = torch.empty_like(P.k_all)
    for c, row_off, start, counts in plan:
        for s in range(S):
            if counts[s] == 0:
                continue
            pos = torch.arange(int(start[s]), int(c[s]), device=dev)
            a, b = int(row_off[s]), int(row_off[s] + counts[s])
            for layer in range(L):
                k, v = synth.context_rows(w.seed, seq_ids[s], layer, pos, w.kv_row, w.sigma, device=dev)
                P.k_all[layer, a:b] = k
                P.v_all[layer, a:b] = v
    P.plan = plan
    P.q, P.kn, P.vn = [], [], []
    for layer in range(L):
        P.q.append(torch.stack([synth.query_block(w.seed, 0, sid, layer, w.q_len, w.n_head, w.head_dim,
                                                  w.sigma, device=dev) for sid in seq_ids]))
        kn, vn = zip(*[synth.noise_rows(w.seed, 0, sid, layer, w.q_len, w.kv_row, w.sigma, device=dev)
                       for sid in seq_ids])
        P.kn.append(torch.stack(kn))
        P.vn.append(torch.stack(vn))
    P.o = [torch.empty((S, w.q_len, w.n_head, w.head_dim), dtype=torch.float32, device=dev)
           for _ in range(L)]
    return P


def visible_rows(w, committed, mask):
    """Visible K/V slot rows of one attention launch (summed over sequences)."""
    tot = 0
    for c in committed:
        win = min(int(c), w.cap)
        if mask == "swa":
            win = min(win, w.swa_window)
        tot += win + w.q_len
    return tot


def shard_sequences(rank: int, world: int, n_seq: int):
    """Weak scaling: every rank owns n_seq independent rings of its own, numbered
    rank * n_seq + s in the seeded generator (no data is exchanged between ranks)."""
    return [rank * n_seq + s for s in range(n_seq)]


def max_over_ranks(value: float, dist, device=None) -> float:
    """The job's time is its slowest rank's time."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _workload(args):
    import synth
    w = synth.workload(args.workload)
    if args.mask == "swa" and not w.swa_window:
        w = synth.workload(args.workload, swa_window=2048)
    if args.n_seq:
        w = synth.workload(args.workload, n_seq=args.n_seq, swa_window=w.swa_window,
                           name=w.name.replace(f"_s{w.n_seq}_", f"_s{args.n_seq}_"))
    return w


class StepBench:
    """One workload on the GPU: its prepared inputs, the ring factory and the timed loop.
    The L2 is flushed between steps when the ring would fit in it: an untimed 512 MiB
    write, then an untimed read of another 512 MiB, so the timed kernels find neither
    useful lines nor the flush's dirty lines (whose write-back they would otherwise pay
    for); larger rings are read from HBM anyway."""

    def __init__(self, w, kind, args, dev, rank, n_steps):
        import torch
        self.w, self.kind, self.args, self.dev = w, kind, args, dev
        self.stream = torch.cuda.current_stream()
        self.P = prepare(w, n_steps, rank, dev)
        r = self.new_ring()
        self.g = r.geometry
        r.close()
        self.flush = self.g["cache_bytes"] * w.n_seq < 2 * L2_BYTES
        self.flush_buf = (torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
                          if self.flush else None)
        self.flush_rd = (torch.zeros(128 * 1024 * 1024, dtype=torch.int32, device=dev)
                         if self.flush else None)

    def new_ring(self, prefill=True):
        import torch
        from speculative_decoding_draft_kv_gb300 import ring as R
        w, a, P = self.w, self.args, self.P
        r = R.Ring(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer, w.rope_theta,
                   n_seq=w.n_seq, swa_window=w.swa_window, tiles_per_split=a.tiles_per_split,
                   max_cluster=a.max_cluster, kv_format=a.kv_format, step_split=a.step_split)
        if prefill:
            c, row_off, start, _ = P.plan[0]             # prefill (bulk path), untimed
            r.begin_step(c, P.k_all, P.v_all, row_off, start, self.stream)
            torch.cuda.synchronize()
        return r

    def step_graph(self, r, t):
        P = self.P
        c, row_off, start, _ = P.plan[t]
        r.step(c, P.k_all, P.v_all, row_off, start, self.kind, P.q, P.kn, P.vn, P.o, self.stream)

    def step_calls(self, r, t):
        P = self.P
        c, row_off, start, _ = P.plan[t]
        r.begin_step(c, P.k_all, P.v_all, row_off, start, self.stream)
        for layer in range(self.w.n_layer):
            r.attend(layer, self.kind, P.q[layer], P.kn[layer], P.vn[layer], P.o[layer], self.stream)

    def timed_loop(self, r, step, t0, n):
        import torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        # an untimed ~1 ms spin first lets the host queue steps ahead of the device, so a
        # host hiccup never leaves the device idle inside a timed step
        torch.cuda._sleep(2_000_000)
        for j in range(n):
            a, b = evs[j]
            a.record(self.stream)
            step(r, t0 + j)
            b.record(self.stream)
            if self.flush:
                self.flush_buf.fill_(j & 0xFF)
                self.flush_rd.amax()
        return evs

    @staticmethod
    def ms_of(evs):
        return sum(a.elapsed_time(b) for a, b in evs)

    def row_bytes(self):
        # bytes a slot row holds: F16 two per value; q8_0 34 per 32 values (codes + scale)
        return self.w.kv_row * (34 / 32 if self.args.kv_format == "q8_0" else 2)

    def attend_bytes(self, committed):
        """Algorithmic bytes of one layer's attention launch: every visible K/V slot row
        once, the queries and the outputs (F32)."""
        w = self.w
        qo = 2 * w.n_seq * w.n_head * w.q_len * w.head_dim * 4
        return visible_rows(w, committed, self.kind) * self.row_bytes() * 2 + qo

    def measure(self, K, W, dist, sampler=None, keep_ring=False):
        """W warm-up steps, then exactly K timed ring_step calls with CUDA events around each,
        the attention kernel's device clock on.  Returns the figures and, when asked, the
        ring (state after the last timed step)."""
        import numpy as np
        import torch
        r = self.new_ring()
        r.clock_enable(True)
        self.timed_loop(r, self.step_graph, 1, W)
        torch.cuda.synchronize()
        r.clock_read()                                  # forget the warm-up launches
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        if sampler:
            sampler.start()
        launches0 = r.launch_count()
        evs = self.timed_loop(r, self.step_graph, 1 + W, K)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        clocks = sampler.stop() if sampler else None
        clock_ms, clock_n = r.clock_read()
        out = {
            "ms_per_step": max_over_ranks(self.ms_of(evs), dist, self.dev) / K,
            "launches": r.launch_count() - launches0,
            "clocks": clocks,
            "clock_ms": clock_ms, "clock_launches": clock_n,
            "last_step": W + K,
        }
        assert r.device_error() == 0
        persistent = self.g["step_split"] > 0
        per_layer = [self.attend_bytes(self.P.plan[1 + W + j][0]) for j in range(K)]
        out["alg_bytes_per_launch"] = float(np.mean(per_layer)) * (self.w.n_layer if persistent else 1)
        out["kernel"] = "k_attend_step" if persistent else "k_attend"
        out["launches_per_step"] = 1 if persistent else self.w.n_layer
        out["step_kv_bytes"] = float(np.mean([visible_rows(self.w, self.P.plan[1 + W + j][0], self.kind)
                                              for j in range(K)])) * self.row_bytes() * 2 * self.w.n_layer
        if keep_ring:
            out["ring"] = r
        else:
            r.close()
        return out

    def roofline(self, m, peak, peak_kind, traffic=None):
        launch_ms = m["clock_ms"] / max(m["clock_launches"], 1)
        achieved = m["alg_bytes_per_launch"] / (launch_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "kernel": m["kernel"],
                "peak_source": f"{peak_kind} hbm_gbs",
                "alg_bytes_per_launch": m["alg_bytes_per_launch"], "launch_ms": launch_ms,
                "launches_per_step": m["launches_per_step"],
                "timing": "device clock of every launch inside the timed graph replays "
                          "(globaltimer: earliest CTA past its grid dependency to the last CTA's "
                          "exit), averaged over the timed steps"}


EXTRA_CONFIGS = [(5, "full"), (4, "full"), (4, "swa")]


def run_gb300(args):
    import numpy as np
    import torch

    import synth
    from speculative_decoding_draft_kv_gb300 import build as B
    from speculative_decoding_draft_kv_gb300 import ring as R

    rank, world, local = _dist_env()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    B.build()
    w = _workload(args)
    K, W = args.steps, args.warmup
    kind = args.mask
    sb = StepBench(w, kind, args, dev, rank, K + W)
    P, g = sb.P, sb.g
    stream = sb.stream
    peak, peak_kind = _peaks()
    q8 = args.kv_format == "q8_0"

    # ---- pass 1: the step graph; warm-up, then exactly K timed steps ----
    sampler = ClockSampler(f"GPU-{torch.cuda.get_device_properties(dev).uuid}") if rank == 0 else None
    head = sb.measure(K, W, dist, sampler, keep_ring=True)
    head_ring = head.pop("ring")
    ms_per_step = head["ms_per_step"]
    tr = NCU_TRAFFIC.get(w.name + ("_q8_0" if q8 else "") + ("_step" if g["step_split"] > 0 else ""))
    src = "step_kernels.cu" if g["step_split"] > 0 else "attn_kernels.cu"
    traffic = tr["bytes"] if tr and tr.get("kernel") == _kernel_source_hash(src) else None
    roof = sb.roofline(head, peak, peak_kind, traffic)

    # ---- pass 2: the same steps as separate calls (begin_step + attend per layer) ----
    n2 = min(K + W, 400)
    ring = sb.new_ring()
    evs = sb.timed_loop(ring, sb.step_calls, 1, n2)
    torch.cuda.synchronize()
    ms_calls = max_over_ranks(sb.ms_of(evs), dist, dev) / n2
    ring.close()

    # ---- pass 3: separate calls with events around every kernel launch (kernel shares) ----
    ring = sb.new_ring()
    R.ring_profile_enable(ring.h, True)
    sb.timed_loop(ring, sb.step_calls, 1, n2)
    torch.cuda.synchronize()
    prof = R.ring_profile_read(ring.h)
    R.ring_profile_enable(ring.h, False)
    ring.close()
    shares = {k: v["total_ms"] for k, v in prof.items() if k != "step_graph"}
    tot = sum(shares.values()) or 1.0
    shares = {k: round(v / tot, 4) for k, v in shares.items()}
    roof["kernel_time_share_separate_calls"] = shares
    row_bytes = sb.row_bytes()

    # ---- pass 4: end to end through ring_step with host buffers: every step copies its
    # new rows, queries and noise rows from pinned host memory and reads every layer's
    # output back ----
    e2e_obj = None
    if not args.no_e2e:
        # The step's inputs live in one device buffer and its outputs in another (views at
        # 256-byte offsets), so a step is two host-to-device copies -- its new rows, then
        # the queries and noise rows of every layer -- and one device-to-host copy of every
        # layer's output, from and to pinned host buffers of the same layout.
        n4 = min(K + W, 400)
        R_max = max(1, max(int(P.plan[t][3].sum()) for t in range(1, 1 + n4)))
        Lw = w.n_layer

        def carve(spec, device=None, pin=False):
            """One uint8 buffer holding tensors of the given (shape, dtype), 256-byte aligned."""
            offs, tot = [], 0
            for shape, dt in spec:
                nb = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
                offs.append(tot)
                tot += (nb + 255) // 256 * 256
            buf = (torch.empty(tot, dtype=torch.uint8, device=device) if device is not None
                   else torch.empty(tot, dtype=torch.uint8, pin_memory=pin))
            views = [buf[o:o + int(np.prod(sh)) * torch.empty((), dtype=dt).element_size()]
                     .view(dt).view(sh) for o, (sh, dt) in zip(offs, spec)]
            return buf, views

        rows_spec = [((Lw, R_max, w.kv_row), torch.float16)] * 2
        in_spec = [(tuple(x.shape), x.dtype) for l in range(Lw) for x in (P.q[l], P.kn[l], P.vn[l])]
        out_spec = [(tuple(o.shape), o.dtype) for o in P.o]
        d_rows, (k_stage, v_stage) = carve(rows_spec, device=dev)
        d_in, dv_in = carve(in_spec, device=dev)
        d_out, dv_out = carve(out_spec, device=dev)
        q_e = dv_in[0::3]
        kn_e = dv_in[1::3]
        vn_e = dv_in[2::3]
        host_rows = []
        for t in range(1, 1 + n4):
            c, row_off, start, counts = P.plan[t]
            n = int(counts.sum())
            hbuf, (hk, hv) = carve(rows_spec, pin=True)
            hbuf.zero_()
            if n:
                a0 = int(row_off[0])
                hk[:, :n] = P.k_all[:, a0:a0 + n].cpu()
                hv[:, :n] = P.v_all[:, a0:a0 + n].cpu()
            host_rows.append((hbuf, (row_off - row_off[0]).astype(np.int64)))
        h_in, hv_in = carve(in_spec, pin=True)
        for l in range(Lw):
            hv_in[3 * l].copy_(P.q[l].cpu())
            hv_in[3 * l + 1].copy_(P.kn[l].cpu())
            hv_in[3 * l + 2].copy_(P.vn[l].cpu())
        h_out, _ = carve(out_spec, pin=True)
        h2d_bytes = 2 * k_stage.numel() * 2 + sum(x.numel() * 4 + y.numel() * 2 + z.numel() * 2
                                                  for x, y, z in zip(q_e, kn_e, vn_e))
        d2h_bytes = sum(o.numel() * 4 for o in dv_out)

        def step_e2e(r, t):
            hbuf, rel_off = host_rows[t - 1]
            d_rows.copy_(hbuf, non_blocking=True)
            d_in.copy_(h_in, non_blocking=True)
            c, _, start, _ = P.plan[t]
            r.step(c, k_stage, v_stage, rel_off, start, kind, q_e, kn_e, vn_e, dv_out, stream)
            h_out.copy_(d_out, non_blocking=True)

        ring = sb.new_ring()
        sb.timed_loop(ring, step_e2e, 1, min(W, n4))        # warm-up (captures the graphs)
        torch.cuda.synchronize()
        ring.close()
        ring = sb.new_ring()
        evs = sb.timed_loop(ring, step_e2e, 1, n4)
        torch.cuda.synchronize()
        ring.close()
        e2e_ms = max_over_ranks(sb.ms_of(evs), dist, dev) / n4
        e2e_obj = {"value": 1000.0 / e2e_ms * world, "unit": UNIT,
                   "h2d_bytes_per_step": int(h2d_bytes), "d2h_bytes_per_step": int(d2h_bytes),
                   "steps": n4, "api": "ring_step",
                   "copies_per_step": "2 host-to-device (the new rows; every layer's queries and "
                                      "noise rows), 1 device-to-host (every layer's output), "
                                      "pinned host buffers"}
    # ---- pass 5: the step with the context rows made by the producer from fused
    # features (ring_begin_step_features + ring_attend per layer), and the producer
    # kernel's own roofline ----
    prod_obj = None
    n_feat_rows = int(sum(int(P.plan[t][3].sum()) for t in range(len(P.plan))))
    if args.producer_hidden > 0 and n_feat_rows * args.producer_hidden * 2 <= (1 << 30):
        H = args.producer_hidden
        ws = [synth.producer_weights(w.seed, l, w.kv_row, H, w.head_dim, device=dev)
              for l in range(w.n_layer)]
        wk = torch.stack([x[0] for x in ws]).contiguous()
        wv = torch.stack([x[1] for x in ws]).contiguous()
        kn = torch.stack([x[2] for x in ws]).contiguous()
        del ws
        feat_all = torch.empty((max(n_feat_rows, 1), H), dtype=torch.float16, device=dev)
        seq_ids = shard_sequences(rank, world, w.n_seq)
        for c, row_off, start, counts in P.plan:
            for s_ in range(w.n_seq):
                if counts[s_]:
                    a = int(row_off[s_])
                    feat_all[a:a + int(counts[s_])] = synth.feature_rows(
                        w.seed, seq_ids[s_], torch.arange(int(start[s_]), int(c[s_]), device=dev),
                        H, w.sigma, device=dev)

        def prod_ring():
            r = R.Ring(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer, w.rope_theta,
                       n_seq=w.n_seq, swa_window=w.swa_window, tiles_per_split=args.tiles_per_split,
                       max_cluster=args.max_cluster, kv_format=args.kv_format)
            r.set_producer(H, 1e-6, wk, wv, kn)
            c, row_off, start, _ = P.plan[0]
            r.begin_step_features(c, feat_all, row_off, start, stream)
            torch.cuda.synchronize()
            return r

        def step_prod(r, t):
            c, row_off, start, _ = P.plan[t]
            r.begin_step_features(c, feat_all, row_off, start, stream)
            for layer in range(w.n_layer):
                r.attend(layer, kind, P.q[layer], P.kn[layer], P.vn[layer], P.o[layer], stream)

        n5 = min(K + W, 400)
        ring = prod_ring()
        ring.clock_enable(True)
        sb.timed_loop(ring, step_prod, 1, min(W, n5))
        torch.cuda.synchronize()
        ring.clock_read("produce")                      # forget the warm-up launches
        evs = sb.timed_loop(ring, step_prod, 1 + min(W, n5), n5 - min(W, n5))
        torch.cuda.synchronize()
        ms_prod = max_over_ranks(sb.ms_of(evs), dist, dev) / max(1, n5 - min(W, n5))
        clk_ms, clk_n = ring.clock_read("produce")
        assert ring.device_error() == 0
        ring.close()
        ring = prod_ring()
        R.ring_profile_enable(ring.h, True)
        sb.timed_loop(ring, step_prod, 1, n5)
        torch.cuda.synchronize()
        pp = R.ring_profile_read(ring.h)
        ring.close()
        pr = pp["produce"]
        prod_ms_isolated = pr["total_ms"] / max(pr["launches"], 1)
        prod_ms = clk_ms / max(clk_n, 1)
        rows = float(np.mean([int(P.plan[1 + j][3].sum()) for j in range(n5)
                              if int(P.plan[1 + j][3].sum()) > 0] or [0]))
        prod_bytes = (2 * w.n_layer * w.kv_row * H * 2 + rows * H * 2
                      + rows * w.n_layer * 2 * row_bytes)
        prod_ach = prod_bytes / (prod_ms * 1e-3) / 1e9
        ptr = PRODUCE_TRAFFIC.get(w.name + ("_q8_0" if q8 else ""))
        prod_traffic = (ptr["bytes"] if ptr and H == 4096
                        and ptr.get("kernel") == _kernel_source_hash("produce_kernels.cu") else None)
        prod_obj = {
            "value": 1000.0 / ms_prod * world, "unit": UNIT, "ms_per_step": ms_prod,
            "steps": n5 - min(W, n5), "hidden": H,
            "api": "ring_begin_step_features + ring_attend per layer",
            "roofline": {"bound": "hbm", "achieved": prod_ach, "peak": peak, "unit": "GB/s",
                         "frac": prod_ach / peak, "traffic": prod_traffic, "kernel": "k_produce",
                         "alg_bytes_per_launch": prod_bytes, "launch_ms": prod_ms,
                         "rows_per_launch": rows,
                         "unit_bytes": "W_k and W_v of every layer + feature rows + K/V rows written",
                         "timing": "device clock of every producer launch inside the timed steps "
                                   "(globaltimer: earliest CTA past its grid dependency to the last "
                                   "CTA's exit; the first 4 weight tiles of each CTA are fetched "
                                   "before the dependency, overlapping the previous kernel)",
                         "launch_ms_isolated": prod_ms_isolated,
                         "frac_isolated": prod_bytes / (prod_ms_isolated * 1e-3) / 1e9 / peak,
                         "isolated": "CUDA events around each launch, launches serialised "
                                     "(no programmatic overlap), launch latency included"},
        }
        # ---- pass 6: the page's legacy path for comparison -- the whole window produced
        # again every step (ring_recompute_window + ring_attend per layer); one sequence ----
        if w.n_seq == 1:
            start0 = int(P.plan[0][2][0])

            def step_legacy(r, t):
                c = P.plan[t][0]
                lo = int(c[0]) - min(int(c[0]), w.cap)
                r.recompute_window(c, feat_all, [lo - start0], [lo], stream)
                for layer in range(w.n_layer):
                    r.attend(layer, kind, P.q[layer], P.kn[layer], P.vn[layer], P.o[layer], stream)

            n6 = min(K + W, 100)
            ring = prod_ring()
            ring.clock_enable(True)
            sb.timed_loop(ring, step_legacy, 1, min(W, n6))
            torch.cuda.synchronize()
            ring.clock_read("produce")                  # forget the warm-up launches
            evs = sb.timed_loop(ring, step_legacy, 1 + min(W, n6), n6 - min(W, n6))
            torch.cuda.synchronize()
            ms_leg = max_over_ranks(sb.ms_of(evs), dist, dev) / max(1, n6 - min(W, n6))
            lclk_ms, lclk_n = ring.clock_read("produce")
            assert ring.device_error() == 0
            ring.close()
            ring = prod_ring()                 # a fresh ring: committed never goes back
            R.ring_profile_enable(ring.h, True)
            sb.timed_loop(ring, step_legacy, 1, min(20, n6))
            torch.cuda.synchronize()
            pl = R.ring_profile_read(ring.h)["produce"]
            ring.close()
            rows6 = min(int(P.plan[1][0][0]), w.cap)
            leg_ms_isolated = pl["total_ms"] / max(pl["launches"], 1)
            leg_ms = lclk_ms / max(lclk_n, 1)
            leg_flops = 2.0 * rows6 * (2 * w.kv_row * w.n_layer) * H
            ltr = PRODUCE_TRAFFIC.get(w.name + "_legacy" + ("_q8_0" if q8 else ""))
            tpeak, tpeak_kind = _tensor_peak()
            prod_obj["legacy_recompute"] = {
                "value": 1000.0 / ms_leg * world, "unit": UNIT, "ms_per_step": ms_leg,
                "steps": n6 - min(W, n6), "rows_per_step": rows6,
                "produce_ms": leg_ms, "produce_ms_isolated": leg_ms_isolated,
                "roofline": {"bound": "tensor", "achieved": leg_flops / (leg_ms * 1e-3) / 1e12,
                             "peak": tpeak, "unit": "TFLOP/s",
                             "frac": leg_flops / (leg_ms * 1e-3) / 1e12 / tpeak,
                             "kernel": "k_produce_tc (tcgen05, accumulators in tensor memory)",
                             "flops_per_launch": leg_flops,
                             "peak_source": f"{tpeak_kind} bf16_tflops (burst; F16 has the same "
                                            "nominal dense rate)",
                             "traffic": (ltr["bytes"] if ltr and H == 4096 and ltr.get("kernel") ==
                                         _kernel_source_hash("produce_tc.cu") else None),
                             "timing": "device clock of every producer launch inside the timed "
                                       "steps (earliest CTA past its grid dependency to the "
                                       "last CTA's exit)",
                             "frac_isolated": leg_flops / (leg_ms_isolated * 1e-3) / 1e12 / tpeak},
                "api": "ring_recompute_window + ring_attend per layer (page section 1.6 fallback)"}
        # ---- pass 7: the whole draft step (ring_draft_step): the producer, the begin-step
        # kernel, then per layer the noise-block Q/K/V projections of its hidden states and
        # its attention (every layer full mask here) ----
        qws = [synth.query_weights(w.seed, l, w.n_head * w.head_dim, H, w.head_dim, device=dev)
               for l in range(w.n_layer)]
        wq = torch.stack([x[0] for x in qws]).contiguous()
        qn = torch.stack([x[1] for x in qws]).contiguous()
        del qws
        noise_h = torch.stack([torch.stack([synth.noise_hidden(w.seed, 0, sid, l, w.q_len, H, w.sigma,
                                                               device=dev) for sid in seq_ids])
                               for l in range(w.n_layer)]).contiguous()
        pattern = [kind] * w.n_layer

        def draft_ring():
            r = prod_ring()
            r.set_producer(H, 1e-6, wk, wv, kn, wq, qn)
            return r

        def step_draft(r, t):
            c, row_off, start, _ = P.plan[t]
            r.draft_step(c, feat_all, row_off, start, noise_h, pattern, P.o, stream)

        n7 = min(K + W, 400)
        ring = draft_ring()
        ring.clock_enable(True)
        sb.timed_loop(ring, step_draft, 1, min(W, n7))
        torch.cuda.synchronize()
        for kind_ in ("attend", "produce", "project"):
            ring.clock_read(kind_)                      # forget the warm-up launches
        evs = sb.timed_loop(ring, step_draft, 1 + min(W, n7), n7 - min(W, n7))
        torch.cuda.synchronize()
        n7t = max(1, n7 - min(W, n7))
        ms_draft = max_over_ranks(sb.ms_of(evs), dist, dev) / n7t
        dclk = {kind_: ring.clock_read(kind_) for kind_ in ("attend", "produce", "project")}
        assert ring.device_error() == 0
        ring.close()
        ring = draft_ring()
        R.ring_profile_enable(ring.h, True)
        sb.timed_loop(ring, step_draft, 1, min(n7, 100))
        torch.cuda.synchronize()
        pd = R.ring_profile_read(ring.h)
        ring.close()
        n_prof = min(n7, 100)
        nrow = w.n_seq * w.q_len
        proj_bytes = (wq.shape[1] + 2 * w.kv_row) * H * 2 + nrow * H * 2 + nrow * (
            w.n_head * w.head_dim * 4 + 2 * w.kv_row * 2)
        proj_ms = dclk["project"][0] / max(dclk["project"][1], 1)
        proj_ach = proj_bytes / (proj_ms * 1e-3) / 1e9
        prod_obj["draft_step"] = {
            "value": 1000.0 / ms_draft * world, "unit": UNIT, "ms_per_step": ms_draft,
            "steps": n7 - min(W, n7), "pattern": pattern,
            "device_clock_ms_per_step": {k: v[0] / n7t for k, v in dclk.items()},
            "projection_roofline": {
                "bound": "hbm", "achieved": proj_ach, "peak": peak, "unit": "GB/s",
                "frac": proj_ach / peak, "kernel": "k_produce (noise rows)",
                "alg_bytes_per_launch": proj_bytes, "launch_ms": proj_ms,
                "unit_bytes": "W_q, W_k, W_v of one layer + its hidden-state rows + Q (F32), "
                              "K, V (F16) rows written",
                "timing": "device clock of every projection launch inside the timed steps"},
            "kernel_ms_per_step_isolated": {k: v["total_ms"] / n_prof for k, v in pd.items()
                                            if k in ("produce", "begin", "attend", "combine")},
            "api": "ring_draft_step (producer + begin + per layer: noise Q/K/V projection, attention)"}
        del wq, qn, noise_h
        del feat_all, wk, wv, kn


    # ---- the roofline workloads of the method (cap 32768 x 16 sequences; cap 4096 x 64
    # sequences with mask_full and with mask_swa, window 2048): the same measurement ----
    extras = []
    if world == 1 and not args.no_extra_configs:
        del sb
        torch.cuda.empty_cache()
        for wid, xkind in EXTRA_CONFIGS:
            xw = synth.workload(wid)
            Kx, Wx = min(K, args.extra_steps), 3
            xsb = StepBench(xw, xkind, args, dev, rank, Kx + Wx)
            xm = xsb.measure(Kx, Wx, None, keep_ring=True)
            xring = xm.pop("ring")
            xtr = NCU_TRAFFIC.get(xw.name + ("_q8_0" if q8 else "") if xkind == "full" else None)
            xroof = xsb.roofline(xm, peak, peak_kind,
                                 xtr["bytes"] if xtr and xtr.get("kernel") == _kernel_source_hash() else None)
            extras.append({"workload": xw.name, "mask": xkind, "value": 1000.0 / xm["ms_per_step"],
                           "unit": UNIT, "ms_per_step": xm["ms_per_step"], "steps": Kx, "warmup": Wx,
                           "step_kv_gbs": xm["step_kv_bytes"] / (xm["ms_per_step"] * 1e-3) / 1e9,
                           "l2": ("flushed between steps" if xsb.flush else "inputs larger than L2"),
                           "split": {k: xsb.g[k] for k in ("tiles_per_split", "n_splits", "cluster",
                                                           "groups", "step_split")},
                           "roofline": xroof, "_ring": xring, "_plan": xsb.P.plan,
                           "_last": xm["last_step"], "_w": xw})
            del xsb
            torch.cuda.empty_cache()

    cpu = None
    state = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle leg: the oracle timed on the host cores, and its bookkeeping (slot map,
        # masks, tile flags) carried through the same commits the timed steps made and
        # compared bit for bit with the GPU ring's final state
        cpu = cpu_baseline(w, kind, n_steps=args.cpu_steps, kv_format=args.kv_format)
        state = state_check(w, kind, P.plan, head["last_step"], head_ring)
        for x in extras:
            n_x = 1 if x["_w"].cap > 8192 else 2
            x["cpu_baseline"] = cpu_baseline(x["_w"], x["mask"], n_steps=n_x, kv_format=args.kv_format)
            x["state_check"] = state_check(x["_w"], x["mask"], x["_plan"], x["_last"], x["_ring"],
                                           seqs=[0, x["_w"].n_seq // 2, x["_w"].n_seq - 1])
    head_ring.close()
    for x in extras:
        x.pop("_ring").close()
        for k in ("_plan", "_last", "_w"):
            x.pop(k)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": 1000.0 / ms_per_step * world,
            "unit": UNIT,
            "n_gpus": world,
            "steps": K,
            "warmup": W,
            "ms_per_step": ms_per_step,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "q8_0 slots, f16 mma, f32 accumulate" if q8 else "f16",
            "data": "synthetic (seeded counter-based generator; the with_producer pass uses "
                    "seeded random-init projection weights)",
            "config": {
                "workload": w.name, "cap": w.cap, "q_len": w.q_len, "n_seq": w.n_seq,
                "n_layer": w.n_layer, "head_dim": w.head_dim, "n_head_kv": w.n_head_kv,
                "n_head": w.n_head, "mask": kind, "kv_format": args.kv_format,
                "kv_total": g["kv_total"],
                "tiles_per_split": g["tiles_per_split"], "n_splits": g["n_splits"],
                "cluster": g["cluster"], "groups": g["groups"], "step_split": g["step_split"],
                "l2": ("flushed between steps (untimed 512 MiB write, then 512 MiB read)" if sb_flush(g, w)
                       else "inputs larger than L2"),
                "api": "ring_step (one CUDA graph per step)",
                "parallelism": f"independent rings x{world}",
            },
            "gpu_launches": int(head["launches"]),
            "separate_calls": {"value": 1000.0 / ms_calls * world, "ms_per_step": ms_calls,
                               "api": "ring_begin_step + ring_attend per layer"},
            "with_producer": prod_obj,
            "step_kv_gbs": head["step_kv_bytes"] / (ms_per_step * 1e-3) / 1e9,
            "roofline": roof,
            "configs": extras,
            "clocks": head["clocks"],
            "e2e": e2e_obj,
            "cpu_baseline": cpu,
            "state_check": state,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def sb_flush(g, w):
    return g["cache_bytes"] * w.n_seq < 2 * L2_BYTES


# ----------------------------------------------------------------------------------------
# CPU oracle legs
# ----------------------------------------------------------------------------------------

def _cpu_worker(task):
    """Oracle work of one host process: a static share of the workload's (sequence, layer)
    units, each a one-layer float64 ring of the step-by-step oracle.  Everything the timed
    steps read (prefill, context rows, queries, noise rows) is made first, untimed; then the
    process times begin_step + attention of its units for the sampled steps."""
    w, kind, units, n_steps, kv_format = task
    import time as _t

    import numpy as np
    import torch
    torch.set_num_threads(1)

    import synth
    from oracle import ring_oracle as orc

    # row 0 is the untimed first call (the prefill where the workload has one)
    sched = synth.commit_schedule(w, n_steps + (0 if w.kind in ("decode", "batched", "large") else 1))
    work = []
    for s, layer in units:
        ring = orc.RingOracle(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, 1, w.rope_theta,
                              swa_window=w.swa_window, kv_format=kv_format)

        def rows(a, b):
            k, v = synth.context_rows(w.seed, s, layer, torch.arange(a, b), w.kv_row, w.sigma)
            return k.numpy()[None], v.numpy()[None]

        c0 = int(sched[0, s])
        st, _ = ring.rows_needed(c0)
        ring.begin_step(c0, *rows(st, c0), st)            # prefill, untimed
        steps = []
        nxt = c0
        for t in range(1, sched.shape[0]):
            c = int(sched[t, s])
            st = max(nxt, c - min(c, w.cap))
            q = synth.query_block(w.seed, t, s, layer, w.q_len, w.n_head, w.head_dim, w.sigma).numpy()
            kn, vn = synth.noise_rows(w.seed, t, s, layer, w.q_len, w.kv_row, w.sigma)
            steps.append((c, rows(st, c), st, q, kn.numpy(), vn.numpy()))
            nxt = c
        work.append((ring, steps))
    t0 = _t.perf_counter()
    for j in range(n_steps):
        for ring, steps in work:
            c, (k, v), st, q, kn, vn = steps[j]
            ring.begin_step(c, k, v, st)
            ring.attend(0, q, kn, vn, kind)
    return _t.perf_counter() - t0


def cpu_baseline(w, kind, n_steps, kv_format="f16"):
    """Time the float64 oracle (ring-state route) on the host's cores: the workload's
    (sequence, layer) units are split statically over one process per core (at most one
    per unit); every process runs the same sampled steps of its units, and a step of the
    whole workload takes the slowest process's time."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor

    units = [(s, layer) for s in range(w.n_seq) for layer in range(w.n_layer)]
    cores = max(1, min(os.cpu_count() or 1, len(units)))
    parts = [units[i::cores] for i in range(cores)]
    with ProcessPoolExecutor(cores, mp_context=mp.get_context("spawn")) as ex:
        secs = list(ex.map(_cpu_worker, [(w, kind, part, n_steps, kv_format) for part in parts]))
    sec_per_step = max(secs) / n_steps
    return {"value": 1.0 / sec_per_step, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n_steps} steps x {w.n_seq} sequences x {w.n_layer} layers ({w.name}, "
                      f"mask {kind}): {len(units)} (sequence, layer) units over {cores} processes, "
                      f"slowest process {max(secs):.1f} s; float64 numpy, one thread each; "
                      f"prefill and input generation untimed"}


def _tile_flags(mask, tile):
    """0: no slot of a tile visible to any row; 1: every slot of a full tile visible to
    every row; 2: anything else."""
    import numpy as np
    n_tiles = (mask.shape[1] + tile - 1) // tile
    out = np.zeros(n_tiles, np.uint8)
    for t in range(n_tiles):
        seg = mask[:, t * tile:(t + 1) * tile] == 0
        out[t] = 0 if not seg.any() else (1 if seg.shape[1] == tile and seg.all() else 2)
    return out


def state_check(w, kind, plan, last, ring, seqs=None):
    """The oracle's bookkeeping (slot map and masks of a head_dim-2 ring) carried through
    the commits plan[0 .. last], against the GPU ring's slot_pos, masks and tile flags,
    bit for bit."""
    import numpy as np

    from oracle import ring_oracle as orc

    g = ring.geometry
    kinds = ["full"] + (["swa"] if w.swa_window else [])
    checked = []
    for s in (range(w.n_seq) if seqs is None else seqs):
        book = orc.RingOracle(w.cap, w.q_len, 2, 1, 1, 1, w.rope_theta, swa_window=w.swa_window)
        for t in range(last + 1):
            c = int(plan[t][0][s])
            st, n = book.rows_needed(c)
            z = np.zeros((1, n, 2), np.float16)
            book.begin_step(c, z, z, st)
        if not np.array_equal(ring.slot_pos(s), book.slot_pos.astype(np.int32)):
            return {"ok": False, "failed": f"slot_pos of sequence {s}"}
        for k in kinds:
            want = book.mask(k)
            got = ring.mask(s, k)
            if got.view(np.uint32).tobytes() != want.view(np.uint32).tobytes():
                return {"ok": False, "failed": f"mask {k} of sequence {s}"}
            if not np.array_equal(ring.tile_flags(s, k), _tile_flags(want, g["tile_slots"])):
                return {"ok": False, "failed": f"tile flags {k} of sequence {s}"}
        checked.append(s)
    return {"ok": True, "steps": last, "sequences": checked, "masks": kinds,
            "what": "slot_pos, masks and tile flags after the timed steps, bit for bit"}


def run_reference(args):
    rank, world, _ = _dist_env()
    if rank != 0:
        return
    w = _workload(args)
    n = max(1, min(args.steps + args.warmup, args.ref_steps))
    cpu = cpu_baseline(w, args.mask, n_steps=n, kv_format=args.kv_format)
    line = {
        "impl": "reference",
        "metric": METRIC, "value": cpu["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / cpu["value"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": w.name, "cap": w.cap, "q_len": w.q_len, "n_seq": w.n_seq,
                   "n_layer": w.n_layer, "mask": args.mask, "kv_format": args.kv_format},
        "cpu_baseline": cpu,
        "e2e": {"value": cpu["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    # Every oracle process runs one thread (the oracle legs spread over processes): keep
    # numpy's BLAS at one thread.  Set before numpy or torch is first imported (inherited
    # by the spawned oracle processes); the GPU path does not use them.
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(var, "1")
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", type=int, default=2, choices=[2, 3, 4, 5])
    ap.add_argument("--mask", choices=["full", "swa"], default="full")
    ap.add_argument("--tiles-per-split", type=int, default=0)
    ap.add_argument("--max-cluster", type=int, default=0)
    ap.add_argument("--n-seq", type=int, default=0, help="override the workload's sequence count")
    ap.add_argument("--step-split", type=int, default=0,
                    help="ring_step attention: 0 one launch per layer, -1 the persistent "
                         "whole-step kernel with the widest cluster, >0 its cluster size")
    ap.add_argument("--cpu-steps", type=int, default=100,
                    help="steps of the headline workload the oracle leg times")
    ap.add_argument("--ref-steps", type=int, default=200,
                    help="at most this many steps for the reference arm (the oracle)")
    ap.add_argument("--extra-steps", type=int, default=40,
                    help="timed steps of each of the method's other roofline workloads")
    ap.add_argument("--no-extra-configs", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kv-format", choices=["f16", "q8_0"], default="f16",
                    help="slot format of the ring (q8_0: 32-value blocks, codes + F16 scale)")
    ap.add_argument("--producer-hidden", type=int, default=4096,
                    help="width of the fused features for the producer pass (0: skip it)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gb300(args)


if __name__ == "__main__":
    main()
