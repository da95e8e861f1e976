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
