"""Benchmark of the DFlash draft-KV ring step on GB300 (one JSON line on stdout).

A step is one ring_begin_step for every sequence plus one ring_attend per layer, all
through the C ABI, on a synthetic workload (seeded inputs; no model weights exist for
this path).  Default workload: one sequence, five layers, cap 4096, q_len 8, prefilled
to 8192 committed tokens and then advanced by the page's acceptance histogram.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--workload 2|3|4|5] [--mask full|swa]

Under torchrun every rank runs its own independent rings (weak scaling, no collective on
the data path); rank 0 prints the line with the max-over-ranks time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
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

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the split-KV attention kernel,
# from one ncu capture, keyed by workload; valid only for the kernel source it was taken on.
NCU_TRAFFIC = {
    "steady_decode_cap4096_s1_l5": {"bytes": 17_120_300, "kernel": "a684f3ab371e7c90",
                                    "source": "profiles/attend_cluster_steady_decode_cap4096_s1_l5.md"},
}


# the same for the context-row producer kernel (workload: steady decode, hidden 4096)
PRODUCE_TRAFFIC = {
    "steady_decode_cap4096_s1_l5": {"bytes": 85_043_500, "kernel": "4be0a7000c1f4369",
                                    "source": "profiles/produce_steady_decode_cap4096_s1_l5.md"},
}


def _kernel_source_hash(name: str = "attn_kernels.cu") -> str:
    p = os.path.join(ROOT, "speculative_decoding_draft_kv_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


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
    P = prepare(w, K + W, rank, dev)
    stream = torch.cuda.current_stream()
    kind = args.mask

    def new_ring():
        r = R.Ring(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer, w.rope_theta,
                   n_seq=w.n_seq, swa_window=w.swa_window, tiles_per_split=args.tiles_per_split,
                   max_cluster=args.max_cluster, kv_format=args.kv_format,
                   step_split=args.step_split)
        c, row_off, start, _ = P.plan[0]             # prefill (bulk path), untimed
        r.begin_step(c, P.k_all, P.v_all, row_off, start, stream)
        torch.cuda.synchronize()
        return r

    ring = new_ring()
    g = ring.geometry
    flush = g["cache_bytes"] * w.n_seq < 2 * L2_BYTES
    flush_buf = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev) if flush else None

    def step_graph(r, t):
        c, row_off, start, _ = P.plan[t]
        r.step(c, P.k_all, P.v_all, row_off, start, kind, P.q, P.kn, P.vn, P.o, stream)

    def step_calls(r, t):
        c, row_off, start, _ = P.plan[t]
        r.begin_step(c, P.k_all, P.v_all, row_off, start, stream)
        for layer in range(w.n_layer):
            r.attend(layer, kind, P.q[layer], P.kn[layer], P.vn[layer], P.o[layer], stream)

    def timed_loop(r, step, t0, n, pre=None, post=None):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        # an untimed ~1 ms spin first lets the host queue steps ahead of the device, so a
        # host hiccup never leaves the device idle inside a timed step
        torch.cuda._sleep(2_000_000)
        for j in range(n):
            a, b = evs[j]
            a.record(stream)
            if pre:
                pre(t0 + j)
            step(r, t0 + j)
            if post:
                post(t0 + j)
            b.record(stream)
            if flush:
                flush_buf.fill_(j & 0xFF)
        return evs

    def ms_of(evs):
        return sum(a.elapsed_time(b) for a, b in evs)

    # ---- pass 1: the step graph; warm-up, then exactly K timed steps ----
    timed_loop(ring, step_graph, 1, W)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(f"GPU-{torch.cuda.get_device_properties(dev).uuid}" if rank == 0 else None)
    if rank == 0:
        sampler.start()
    launches0 = ring.launch_count()
    evs = timed_loop(ring, step_graph, 1 + W, K)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches = ring.launch_count() - launches0
    clocks = sampler.stop() if rank == 0 else None
    ms_per_step = max_over_ranks(ms_of(evs), dist, dev) / K
    assert ring.device_error() == 0
    ring.close()

    # ---- pass 2: the same steps as separate calls (begin_step + attend per layer) ----
    n2 = min(K + W, 400)
    ring = new_ring()
    evs = timed_loop(ring, step_calls, 1, n2)
    torch.cuda.synchronize()
    ms_calls = max_over_ranks(ms_of(evs), dist, dev) / n2
    ring.close()

    # ---- pass 3: separate calls with events around every kernel launch ----
    ring = new_ring()
    R.ring_profile_enable(ring.h, True)
    timed_loop(ring, step_calls, 1, n2)
    torch.cuda.synchronize()
    prof = R.ring_profile_read(ring.h)
    R.ring_profile_enable(ring.h, False)
    ring.close()
    attn = prof["attend"]
    attn_ms = attn["total_ms"] / max(attn["launches"], 1)
    vis = float(np.mean([visible_rows(w, P.plan[1 + j][0], kind) for j in range(n2)]))
    q8 = args.kv_format == "q8_0"
    # bytes a slot row holds: F16 two per value; q8_0 34 per 32 values (codes + F16 scale)
    row_bytes = w.kv_row * (34 / 32 if q8 else 2)
    kv_bytes = vis * row_bytes * 2
    q_bytes = w.n_seq * w.n_head * w.q_len * w.head_dim * 4
    o_bytes = w.n_seq * w.n_head * w.q_len * w.head_dim * 4
    alg_bytes = kv_bytes + q_bytes + o_bytes
    peak, peak_kind = _peaks()
    achieved = alg_bytes / (attn_ms * 1e-3) / 1e9
    tr = NCU_TRAFFIC.get(w.name + ("_q8_0" if q8 else ""))
    traffic = tr["bytes"] if tr and tr.get("kernel") == _kernel_source_hash() else None
    shares = {k: v["total_ms"] for k, v in prof.items() if k != "step_graph"}
    tot = sum(shares.values()) or 1.0
    shares = {k: round(v / tot, 4) for k, v in shares.items()}

    # ---- pass 4: end to end through ring_step with host buffers: every step copies its
    # new rows, queries and noise rows from pinned host memory and reads every layer's
    # output back ----
    e2e_obj = None
    if not args.no_e2e:
        n4 = min(K + W, 400)
        R_max = max(1, max(int(P.plan[t][3].sum()) for t in range(1, 1 + n4)))
        k_stage = torch.zeros((w.n_layer, R_max, w.kv_row), dtype=torch.float16, device=dev)
        v_stage = torch.zeros_like(k_stage)
        host_rows = []
        for t in range(1, 1 + n4):
            c, row_off, start, counts = P.plan[t]
            n = int(counts.sum())
            hk = torch.zeros((w.n_layer, R_max, w.kv_row), dtype=torch.float16).pin_memory()
            hv = torch.zeros_like(hk).pin_memory()
            if n:
                a = int(row_off[0])
                hk[:, :n] = P.k_all[:, a:a + n].cpu()
                hv[:, :n] = P.v_all[:, a:a + n].cpu()
            host_rows.append((hk, hv, (row_off - row_off[0]).astype(np.int64)))
        host_in = [(x.cpu().pin_memory(), y.cpu().pin_memory(), z.cpu().pin_memory())
                   for x, y, z in zip(P.q, P.kn, P.vn)]
        host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in P.o]
        h2d_bytes = 2 * k_stage.numel() * 2 + sum(x.numel() * 4 + y.numel() * 2 + z.numel() * 2
                                                  for x, y, z in host_in)
        d2h_bytes = sum(o.numel() * 4 for o in P.o)

        def step_e2e(r, t):
            hk, hv, rel_off = host_rows[t - 1]
            k_stage.copy_(hk, non_blocking=True)
            v_stage.copy_(hv, non_blocking=True)
            for (hq, hkn, hvn), q, kn, vn in zip(host_in, P.q, P.kn, P.vn):
                q.copy_(hq, non_blocking=True)
                kn.copy_(hkn, non_blocking=True)
                vn.copy_(hvn, non_blocking=True)
            c, _, start, _ = P.plan[t]
            r.step(c, k_stage, v_stage, rel_off, start, kind, P.q, P.kn, P.vn, P.o, stream)
            for o, ho in zip(P.o, host_out):
                ho.copy_(o, non_blocking=True)

        ring = new_ring()
        timed_loop(ring, step_e2e, 1, min(W, n4))        # warm-up (captures the graph)
        torch.cuda.synchronize()
        ring.close()
        ring = new_ring()
        evs = timed_loop(ring, step_e2e, 1, n4)
        torch.cuda.synchronize()
        ring.close()
        e2e_ms = max_over_ranks(ms_of(evs), dist, dev) / n4
        e2e_obj = {"value": 1000.0 / e2e_ms * world, "unit": UNIT,
                   "h2d_bytes_per_step": int(h2d_bytes), "d2h_bytes_per_step": int(d2h_bytes),
                   "steps": n4, "api": "ring_step"}

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
                       max_cluster=args.max_cluster)
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
        timed_loop(ring, step_prod, 1, min(W, n5))
        torch.cuda.synchronize()
        evs = timed_loop(ring, step_prod, 1 + min(W, n5), n5 - min(W, n5))
        torch.cuda.synchronize()
        ms_prod = max_over_ranks(ms_of(evs), dist, dev) / max(1, n5 - min(W, n5))
        assert ring.device_error() == 0
        ring.close()
        ring = prod_ring()
        R.ring_profile_enable(ring.h, True)
        timed_loop(ring, step_prod, 1, n5)
        torch.cuda.synchronize()
        pp = R.ring_profile_read(ring.h)
        ring.close()
        pr = pp["produce"]
        prod_ms = pr["total_ms"] / max(pr["launches"], 1)
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
                         "unit_bytes": "W_k and W_v of every layer + feature rows + K/V rows written"},
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
            timed_loop(ring, step_legacy, 1, min(W, n6))
            torch.cuda.synchronize()
            evs = timed_loop(ring, step_legacy, 1 + min(W, n6), n6 - min(W, n6))
            torch.cuda.synchronize()
            ms_leg = max_over_ranks(ms_of(evs), dist, dev) / max(1, n6 - min(W, n6))
            assert ring.device_error() == 0
            ring.close()
            ring = prod_ring()                 # a fresh ring: committed never goes back
            R.ring_profile_enable(ring.h, True)
            timed_loop(ring, step_legacy, 1, min(20, n6))
            torch.cuda.synchronize()
            pl = R.ring_profile_read(ring.h)["produce"]
            ring.close()
            prod_obj["legacy_recompute"] = {
                "value": 1000.0 / ms_leg * world, "unit": UNIT, "ms_per_step": ms_leg,
                "steps": n6 - min(W, n6), "rows_per_step": min(int(P.plan[1][0][0]), w.cap),
                "produce_ms": pl["total_ms"] / max(pl["launches"], 1),
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
        timed_loop(ring, step_draft, 1, min(W, n7))
        torch.cuda.synchronize()
        evs = timed_loop(ring, step_draft, 1 + min(W, n7), n7 - min(W, n7))
        torch.cuda.synchronize()
        ms_draft = max_over_ranks(ms_of(evs), dist, dev) / max(1, n7 - min(W, n7))
        assert ring.device_error() == 0
        ring.close()
        ring = draft_ring()
        R.ring_profile_enable(ring.h, True)
        timed_loop(ring, step_draft, 1, min(n7, 100))
        torch.cuda.synchronize()
        pd = R.ring_profile_read(ring.h)
        ring.close()
        n_prof = min(n7, 100)
        prod_obj["draft_step"] = {
            "value": 1000.0 / ms_draft * world, "unit": UNIT, "ms_per_step": ms_draft,
            "steps": n7 - min(W, n7), "pattern": pattern,
            "kernel_ms_per_step": {k: v["total_ms"] / n_prof for k, v in pd.items()
                                   if k in ("produce", "begin", "attend", "combine")},
            "api": "ring_draft_step (producer + begin + per layer: noise Q/K/V projection, attention)"}
        del wq, qn, noise_h
        del feat_all, wk, wv, kn

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, kind, budget_s=args.cpu_seconds, kv_format=args.kv_format)

    if rank == 0:
        vis_step = visible_rows(w, P.plan[1][0], kind) * row_bytes * 2 * w.n_layer
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
                "cluster": g["cluster"], "groups": g["groups"],
                "l2": ("flushed between steps (512 MiB write, untimed)" if flush
                       else "inputs larger than L2"),
                "api": "ring_step (one CUDA graph per step)",
                "parallelism": f"independent rings x{world}",
            },
            "gpu_launches": int(launches),
            "separate_calls": {"value": 1000.0 / ms_calls * world, "ms_per_step": ms_calls,
                               "api": "ring_begin_step + ring_attend per layer"},
            "with_producer": prod_obj,
            "step_kv_gbs": vis_step / (ms_per_step * 1e-3) / 1e9,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": "k_attend", "peak_source": f"{peak_kind} hbm_gbs",
                         "alg_bytes_per_launch": alg_bytes, "launch_ms": attn_ms,
                         "timing": "CUDA events around each launch on its stream, "
                                   "instrumented repeat of the timed steps as separate calls",
                         "kernel_time_share": shares},
            "clocks": clocks,
            "e2e": e2e_obj,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


# ----------------------------------------------------------------------------------------
# CPU oracle legs
# ----------------------------------------------------------------------------------------

def _oracle_setup(w, kv_format="f16"):
    import numpy as np
    import torch

    import synth
    from oracle import ring_oracle as orc

    sched = synth.commit_schedule(w, 10000)
    S = w.n_seq
    rings = [orc.RingOracle(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer,
                            w.rope_theta, swa_window=w.swa_window, kv_format=kv_format)
             for _ in range(S)]

    def rows(s, a, b):
        ks, vs = [], []
        for layer in range(w.n_layer):
            k, v = synth.context_rows(w.seed, s, layer, torch.arange(a, b), w.kv_row, w.sigma)
            ks.append(k.numpy())
            vs.append(v.numpy())
        return np.stack(ks), np.stack(vs)

    def inputs(t, s):
        out = []
        for layer in range(w.n_layer):
            q = synth.query_block(w.seed, t, s, layer, w.q_len, w.n_head, w.head_dim, w.sigma).numpy()
            kn, vn = synth.noise_rows(w.seed, t, s, layer, w.q_len, w.kv_row, w.sigma)
            out.append((q, kn.numpy(), vn.numpy()))
        return out

    return sched, rings, rows, inputs


def cpu_baseline(w, kind, budget_s=15.0, max_steps=None, kv_format="f16"):
    """Time the float64 oracle (ring-state route) on the host: untimed prefill, then as many
    full steps (begin_step for every sequence + every layer's attention, inputs drawn
    beforehand) as fit in ``budget_s``."""
    import time as _t

    sched, rings, rows, inputs = _oracle_setup(w, kv_format)
    S = w.n_seq
    sample_seqs = min(S, 1)
    for s in range(sample_seqs):
        st, _ = rings[s].rows_needed(int(sched[0, s]))
        k, v = rows(s, st, int(sched[0, s]))
        rings[s].begin_step(int(sched[0, s]), k, v, st)
    done, elapsed = 0, 0.0
    t = 1
    while elapsed < budget_s and (max_steps is None or done < max_steps):
        pre = []
        for s in range(sample_seqs):
            c = int(sched[t, s])
            st, _ = rings[s].rows_needed(c)
            pre.append((c, rows(s, st, c), st, inputs(t, s)))
        t0 = _t.perf_counter()
        for s in range(sample_seqs):
            c, (k, v), st, inp = pre[s]
            rings[s].begin_step(c, k, v, st)
            for layer, (q, kn, vn) in enumerate(inp):
                rings[s].attend(layer, q, kn, vn, kind)
        elapsed += _t.perf_counter() - t0
        done += 1
        t += 1
    # a step of the workload covers all S sequences; the sample covered sample_seqs
    sec_per_step = elapsed / done * (S / sample_seqs)
    return {"value": 1.0 / sec_per_step, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{done} steps x {sample_seqs} of {S} sequences x {w.n_layer} layers "
                      f"({elapsed:.1f} s), scaled to all sequences; float64 numpy, one thread"}


def run_reference(args):
    rank, world, _ = _dist_env()
    if rank != 0:
        return
    w = _workload(args)
    budget = max(5.0, min(150.0, 0.6 * (args.steps + args.warmup)))
    cpu = cpu_baseline(w, args.mask, budget_s=budget, max_steps=args.steps + args.warmup,
                       kv_format=args.kv_format)
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
    # The oracle legs report one host thread: keep numpy's BLAS (and torch's CPU pool) at one
    # thread.  Set before numpy or torch is first imported; the GPU path does not use them.
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
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
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
