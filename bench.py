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
NCU_TRAFFIC = {}


def _kernel_source_hash() -> str:
    p = os.path.join(ROOT, "speculative_decoding_draft_kv_gb300", "csrc", "attn_kernels.cu")
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


def prepare(w, n_steps, mask, rank, dev, pool):
    import numpy as np
    import torch

    import synth

    sched = synth.commit_schedule(w, n_steps)          # row 0: prefill
    P = Prepared()
    P.sched = sched
    S, L = w.n_seq, w.n_layer
    seq_ids = [rank * S + s for s in range(S)]
    # per-step new rows [start, c) for every sequence, concatenated
    next_pos = np.zeros(S, np.int64)
    steps = []
    for t in range(sched.shape[0]):
        c = sched[t]
        win = np.minimum(c, w.cap)
        start = np.maximum(next_pos, c - win)
        counts = (c - start).astype(np.int64)
        n_rows = int(counts.sum())
        row_off = np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int64)
        k_rows = v_rows = None
        if n_rows:
            k_rows = torch.empty((L, n_rows, w.kv_row), dtype=torch.float16, device=dev)
            v_rows = torch.empty_like(k_rows)
            for s in range(S):
                if counts[s] == 0:
                    continue
                pos = torch.arange(int(start[s]), int(c[s]), device=dev)
                a, b = int(row_off[s]), int(row_off[s] + counts[s])
                for layer in range(L):
                    k, v = synth.context_rows(w.seed, seq_ids[s], layer, pos, w.kv_row, w.sigma, device=dev)
                    k_rows[layer, a:b] = k
                    v_rows[layer, a:b] = v
        steps.append((c.copy(), k_rows, v_rows, row_off, start.copy(), int(counts.sum())))
        next_pos = c.copy()
    P.steps = steps
    # a pool of distinct per-step layer inputs (queries and noise rows), cycled
    P.inputs = []
    for j in range(pool):
        per_layer = []
        for layer in range(L):
            q = torch.stack([synth.query_block(w.seed, j, sid, layer, w.q_len, w.n_head, w.head_dim,
                                               w.sigma, device=dev) for sid in seq_ids])
            kn, vn = zip(*[synth.noise_rows(w.seed, j, sid, layer, w.q_len, w.kv_row, w.sigma,
                                            device=dev) for sid in seq_ids])
            per_layer.append((q, torch.stack(kn), torch.stack(vn)))
        P.inputs.append(per_layer)
    P.outputs = [torch.empty((S, w.q_len, w.n_head, w.head_dim), dtype=torch.float32, device=dev)
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
    w = synth.workload(args.workload)
    if args.mask == "swa" and not w.swa_window:
        w = synth.workload(args.workload, swa_window=2048)
    K, W = args.steps, args.warmup
    pool = min(K + W, args.pool)
    P = prepare(w, K + W, args.mask, rank, dev, pool)
    stream = torch.cuda.current_stream()
    kind = args.mask

    def new_ring():
        r = R.Ring(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer, w.rope_theta,
                   n_seq=w.n_seq, swa_window=w.swa_window, tiles_per_split=args.tiles_per_split,
                   max_cluster=args.max_cluster)
        c, k_rows, v_rows, row_off, start, _ = P.steps[0]      # prefill (bulk path), untimed
        r.begin_step(c, k_rows, v_rows, row_off, start, stream)
        torch.cuda.synchronize()
        return r

    ring = new_ring()
    g = ring.geometry
    flush = g["cache_bytes"] * w.n_seq < 2 * L2_BYTES
    flush_buf = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev) if flush else None

    def step(r, t):
        c, k_rows, v_rows, row_off, start, _ = P.steps[t]
        r.begin_step(c, k_rows, v_rows, row_off, start, stream)
        inp = P.inputs[t % pool]
        for layer in range(w.n_layer):
            q, kn, vn = inp[layer]
            r.attend(layer, kind, q, kn, vn, P.outputs[layer], stream)

    def timed_loop(r, t0, n, pre=None, post=None):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
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

    # ---- pass 1: warm-up, then exactly K timed steps ----
    timed_loop(ring, 1, W)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(f"GPU-{torch.cuda.get_device_properties(dev).uuid}" if rank == 0 else None)
    if rank == 0:
        sampler.start()
    launches0 = ring.launch_count()
    evs = timed_loop(ring, 1 + W, K)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches = ring.launch_count() - launches0
    clocks = sampler.stop() if rank == 0 else None
    ms_total = sum(a.elapsed_time(b) for a, b in evs)
    if dist:
        t = torch.tensor([ms_total], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_total = float(t.item())
    ms_per_step = ms_total / K
    assert ring.device_error() == 0
    ring.close()

    # ---- pass 2: the same steps again on a fresh ring, events around each attention launch ----
    n_prof = min(K + W, 400)
    ring = new_ring()
    R.ring_profile_enable(ring.h, True)
    timed_loop(ring, 1, n_prof)
    torch.cuda.synchronize()
    prof = R.ring_profile_read(ring.h)
    R.ring_profile_enable(ring.h, False)
    ring.close()
    attn = prof["attend"]
    attn_ms = attn["total_ms"] / max(attn["launches"], 1)
    vis = float(np.mean([visible_rows(w, P.steps[1 + j][0], kind) for j in range(n_prof)]))
    kv_bytes = vis * w.kv_row * 2 * 2
    q_bytes = w.n_seq * w.n_head * w.q_len * w.head_dim * 2
    o_bytes = w.n_seq * w.n_head * w.q_len * w.head_dim * 4
    alg_bytes = kv_bytes + q_bytes + o_bytes
    peak, peak_kind = _peaks()
    achieved = alg_bytes / (attn_ms * 1e-3) / 1e9
    tr = NCU_TRAFFIC.get(w.name)
    traffic = tr["bytes"] if tr and tr.get("kernel") == _kernel_source_hash() else None
    shares = {k: v["total_ms"] for k, v in prof.items()}
    tot = sum(shares.values()) or 1.0
    shares = {k: round(v / tot, 4) for k, v in shares.items()}

    # ---- pass 3: end to end with host buffers (pinned H2D of each step's rows, queries and
    # noise rows; D2H of every layer's output), on a fresh ring ----
    e2e_obj = None
    if not args.no_e2e:
        n_e2e = min(K + W, 400)
        host_rows = {}
        for t in range(1, 1 + n_e2e):
            _, k_rows, v_rows, _, _, _ = P.steps[t]
            if k_rows is not None:
                host_rows[t] = (k_rows.cpu().pin_memory(), v_rows.cpu().pin_memory())
        host_inp = [[tuple(x.cpu().pin_memory() for x in trip) for trip in per_layer]
                    for per_layer in P.inputs]
        host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in P.outputs]
        h2d = []

        def pre(t):
            nb = 0
            if t in host_rows:
                _, k_rows, v_rows, _, _, _ = P.steps[t]
                k_rows.copy_(host_rows[t][0], non_blocking=True)
                v_rows.copy_(host_rows[t][1], non_blocking=True)
                nb += 2 * host_rows[t][0].numel() * 2
            for layer, trip in enumerate(host_inp[t % pool]):
                for src, dst in zip(trip, P.inputs[t % pool][layer]):
                    dst.copy_(src, non_blocking=True)
                    nb += src.numel() * src.element_size()
            h2d.append(nb)

        def post(t):
            for src, dst in zip(P.outputs, host_out):
                dst.copy_(src, non_blocking=True)

        ring = new_ring()
        evs = timed_loop(ring, 1, n_e2e, pre=pre, post=post)
        torch.cuda.synchronize()
        ring.close()
        e2e_ms = sum(a.elapsed_time(b) for a, b in evs) / n_e2e
        e2e_obj = {"value": 1000.0 / e2e_ms * world, "unit": UNIT,
                   "h2d_bytes_per_step": int(np.mean(h2d)),
                   "d2h_bytes_per_step": int(sum(o.numel() * 4 for o in P.outputs)),
                   "steps": n_e2e}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, kind, budget_s=args.cpu_seconds)

    if rank == 0:
        vis_step = visible_rows(w, P.steps[1][0], kind) * w.kv_row * 4 * w.n_layer
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
            "dtype": "f16",
            "data": "synthetic (seeded counter-based generator; no weights involved)",
            "config": {
                "workload": w.name, "cap": w.cap, "q_len": w.q_len, "n_seq": w.n_seq,
                "n_layer": w.n_layer, "head_dim": w.head_dim, "n_head_kv": w.n_head_kv,
                "n_head": w.n_head, "mask": kind, "kv_total": g["kv_total"],
                "tiles_per_split": g["tiles_per_split"], "n_splits": g["n_splits"],
                "cluster": g["cluster"], "groups": g["groups"],
                "l2": ("flushed between steps (512 MiB write, untimed)" if flush
                       else "inputs larger than L2"),
                "query_pool": pool, "parallelism": f"independent rings x{world}",
            },
            "gpu_launches": int(launches),
            "step_kv_gbs": vis_step / (ms_per_step * 1e-3) / 1e9,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": "k_attend", "peak_source": f"{peak_kind} hbm_gbs",
                         "alg_bytes_per_launch": alg_bytes, "launch_ms": attn_ms,
                         "timing": "CUDA events around each launch on its stream, "
                                   "instrumented repeat of the timed steps",
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

def _oracle_setup(w):
    import numpy as np
    import torch

    import synth
    from oracle import ring_oracle as orc

    sched = synth.commit_schedule(w, 10000)
    S = w.n_seq
    rings = [orc.RingOracle(w.cap, w.q_len, w.head_dim, w.n_head_kv, w.n_head, w.n_layer,
                            w.rope_theta, swa_window=w.swa_window) for _ in range(S)]

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


def cpu_baseline(w, kind, budget_s=15.0, max_steps=None):
    """Time the float64 oracle (ring-state route) on the host: untimed prefill, then as many
    full steps (begin_step for every sequence + every layer's attention, inputs drawn
    beforehand) as fit in ``budget_s``."""
    import time as _t

    sched, rings, rows, inputs = _oracle_setup(w)
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
    import synth
    w = synth.workload(args.workload)
    if args.mask == "swa" and not w.swa_window:
        w = synth.workload(args.workload, swa_window=2048)
    budget = max(5.0, min(150.0, 0.6 * (args.steps + args.warmup)))
    cpu = cpu_baseline(w, args.mask, budget_s=budget, max_steps=args.steps + args.warmup)
    line = {
        "impl": "reference",
        "metric": METRIC, "value": cpu["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / cpu["value"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": w.name, "cap": w.cap, "q_len": w.q_len, "n_seq": w.n_seq,
                   "n_layer": w.n_layer, "mask": args.mask},
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
    ap.add_argument("--pool", type=int, default=64)
    ap.add_argument("--tiles-per-split", type=int, default=0)
    ap.add_argument("--max-cluster", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gb300(args)


if __name__ == "__main__":
    main()
