"""Host logic of the multi-GPU bench path on CPU (gloo, world size 2).

The operator shards by rows with no exchange, so several GPUs run independent
replicas; the only cross-rank steps are the barrier around the timed region
and the max over ranks of the elapsed time (bench.py: barrier, max_over_ranks).
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    got = bench.max_over_ranks(1.5 + rank, world, "cpu")    # rank r "took" 1.5 + r seconds
    bench.barrier(world)
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_world2():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, None) == 3.25
    bench.barrier(1)
