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
        # one rank saw a thermal slowdown: every rank measures again
        ok = {"sm_mhz": 1800.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 9}
        hot = dict(ok, reasons=["sw_power_cap", "sw_thermal_slowdown"])
        again = bench.needs_remeasure(hot if rank == 1 else ok, world, torch.device("cpu"))
        fine = bench.needs_remeasure(ok, world, torch.device("cpu"))
        out[rank] = (bench.rank_seed(7, rank), got, again, fine)
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
    assert out[0][2] and out[1][2] and not out[0][3] and not out[1][3]


def test_remeasure_rule_single_rank():
    import bench
    cpu = torch.device("cpu")
    base = {"sm_mhz": 1650.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 5}
    assert not bench.needs_remeasure(base, 1, cpu)          # power cap: kept and noted
    assert bench.needs_remeasure(dict(base, reasons=["hw_slowdown"]), 1, cpu)
    assert bench.needs_remeasure(dict(base, reasons=["hw_thermal_slowdown"]), 1, cpu)
    # clocks stuck far below the maximum with no reason: a leftover clock lock
    assert bench.needs_remeasure(dict(base, sm_mhz=900.0, reasons=[]), 1, cpu)
    assert not bench.needs_remeasure(dict(base, sm_mhz=1900.0, reasons=[]), 1, cpu)
    assert not bench.needs_remeasure(dict(base, sm_mhz=None, sm_max_mhz=None, reasons=[]), 1,
                                     cpu)
