"""Multi-process host logic of bench.py on CPU (gloo, world size 2): every rank
scans its own seeded batch (weak scaling, no data-path collective) and the
job time is the maximum over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(1.0 + rank, world)          # each rank reports its own time
        seed = bench.rank_seed(100, rank)
        seeds = [None] * world
        dist.all_gather_object(seeds, seed)
        out[rank] = (t, tuple(seeds))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_distinct_seeds():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.0                       # slowest rank decides
    seeds = res[0][1]
    assert len(set(seeds)) == world and seeds[0] == 100       # rank 0 keeps the workload seed


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.rank_seed(7, 0) == 7
