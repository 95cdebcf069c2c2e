"""Multi-rank host logic of bench.py on CPU: world size 2 over gloo.

The layer runs as independent replicas (one per GPU); the job's throughput is
the work of all ranks over the slowest rank's timed region.
"""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env() == (rank, world, rank)
    ms, units = bench.rank_aggregate(10.0 + 5.0 * rank, 1000.0 * (rank + 1), dist)
    q.put((rank, ms, units))
    dist.barrier()
    dist.destroy_process_group()


def test_rank_aggregate_world_size_2_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, units in got:
        assert ms == 15.0           # slowest rank's time
        assert units == 3000.0      # all ranks' work


def test_rank_aggregate_single_process():
    import bench
    assert bench.rank_aggregate(3.0, 7.0, None) == (3.0, 7.0)
