"""Host-side logic of the multi-GPU benchmark path on CPU (gloo, world size 2):
each rank gets its own batch seed, and the reported time is the max over
ranks.  No data-path collective exists to test: ranks score disjoint batches."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        w, r, lr = bench.dist_env()
        assert (w, r, lr) == (world, rank, rank)
        mine = [10.0 + rank, 5.0 - rank, float(rank)]
        got = bench.max_over_ranks(mine, world, torch.device("cpu"))
        out[rank] = (bench.rank_seed(7, rank), got)
    finally:
        dist.destroy_process_group()


def test_two_rank_seeds_and_max_timing():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0][0] != out[1][0]
    assert out[0][1] == out[1][1] == [11.0, 5.0, 1.0]
