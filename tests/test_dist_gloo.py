"""The benchmark's multi-rank host logic on two CPU ranks (gloo): every rank owns its
own independent rings (weak scaling, no data exchanged), and the job's time is the slowest
rank's time."""

import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench._dist_env() == (rank, world, rank)
    ids = bench.shard_sequences(rank, world, 3)
    slowest = bench.max_over_ranks(10.0 * (rank + 1), dist)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, ids, slowest))


def test_two_ranks_shard_and_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict((r, (ids, t)) for r, ids, t in (q.get(timeout=120) for _ in procs))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == [0, 1, 2] and res[1][0] == [3, 4, 5]
    assert res[0][1] == res[1][1] == 20.0


def test_reference_arm_runs_on_rank_zero_only():
    """Under a multi-rank launch the reference arm (the oracle on the host) runs on rank 0
    alone and prints one line; the other ranks exit 0 without work or output."""
    import json
    import subprocess
    base = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()),
                WORLD_SIZE="2")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3"]
    r1 = subprocess.run(cmd, env=dict(base, RANK="1", LOCAL_RANK="1"), capture_output=True,
                        text=True, timeout=120)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = subprocess.run(cmd, env=dict(base, RANK="0", LOCAL_RANK="0"), capture_output=True,
                        text=True, timeout=300)
    assert r0.returncode == 0, r0.stderr[-2000:]
    lines = [x for x in r0.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
