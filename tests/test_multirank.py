"""Multi-process host logic of bench.py on CPU (gloo, world_size 2).

The path has no exchange step, so N GPUs run N independent replicas; what the
ranks share is the timing protocol: a barrier around the timed steps, the
per-step time taken as the max over ranks, and rank 0 alone reporting.
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench

    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # rank r "measured" (r+1) ms per step and a score time of 10 - r ms
    got = bench.reduce_max([float(rank + 1), 10.0 - rank], w, torch.device("cpu"))
    out[rank] = got
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_ranks_take_the_max_over_ranks():
    world = 2
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == [2.0, 10.0]


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import torch
    import bench
    assert bench.reduce_max([1.5, 2.5], 1, torch.device("cpu")) == [1.5, 2.5]
    bench.barrier(1)   # no-op without a process group
