"""bench.py's multi-rank logic (barrier, max-over-ranks time, summed work)
on two gloo ranks on the CPU: replicas only, no data-path collective."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, l = bench.dist_env()
    assert (w, r, l) == (world, rank, rank)
    bench.init_dist(world, "gloo")
    bench.barrier(world)
    t = bench.reduce_max(10.0 + rank, world)           # slowest rank sets the time
    s = bench.reduce_sum(1.5, world)                   # whole-job work
    out[rank] = (t, s)
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == (11.0, 3.0)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25 and bench.reduce_sum(2.0, 1) == 2.0
