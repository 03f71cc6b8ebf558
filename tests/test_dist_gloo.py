"""The multi-rank timing path of bench.py (max elapsed over ranks, sum of units) on CPU with
two gloo ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, lr = bench.dist_env()
    bench.barrier(w)
    el, units = bench.reduce_timing(1.0 + rank, 100.0 * (rank + 1), w)
    q.put((r, w, el, units))
    dist.destroy_process_group()


def test_reduce_timing_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 2, 2.0, 300.0), (1, 2, 2.0, 300.0)]


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_timing(3.5, 42.0, 1) == (3.5, 42.0)
