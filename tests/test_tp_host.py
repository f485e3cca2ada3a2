"""Host logic of the vocab-sharded (tensor-parallel) forward, on CPU: block
boundaries, target ownership, and the partials exchange over a 2-rank gloo
group (each rank's partials land in global chunk order, each row's target
logit comes from the rank that owns its target)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

from rl_post_linear_gb300 import tp


@pytest.mark.parametrize("vocab,parts", [(151936, 1), (151936, 2), (151936, 8), (129280, 4),
                                         (1000, 3), (5000, 4), (1, 2)])
def test_vocab_shards(vocab, parts):
    sh = tp.vocab_shards(vocab, parts)
    assert len(sh) == parts
    pos = 0
    for i, (start, size) in enumerate(sh):
        assert start == pos and start % 1024 == 0 or size == 0
        if i < parts - 1 and size > 0 and start + size < vocab:
            assert size % 1024 == 0
        pos = start + size
    assert pos == vocab
    # the blocks' chunk counts add up to the unsharded count
    assert sum(-(-s // 1024) for _, s in sh) == -(-vocab // 1024)


def test_owner_and_assemble():
    sh = tp.vocab_shards(5000, 3)
    targets = torch.tensor([0, 1023, 1024, 4999, -1, 2500])
    owner = tp.owner_of(targets, sh)
    starts = [s for s, _ in sh]
    for t, o in zip(targets.tolist(), owner.tolist()):
        if t < 0:
            assert o == -1
        else:
            assert starts[o] <= t < starts[o] + sh[o][1]
    n = len(targets)
    # rank r's chunk c holds the value 100 r + c in every element: the assembled partials must
    # list the chunks of rank 0, then rank 1, ..., each rank's in its own chunk order, which for
    # blocks starting on 1024-row boundaries is the global chunk order
    counts = [-(-size // 1024) for _, size in sh]
    assert counts == [1, 2, 2]          # blocks of 1024, 2048 and 1928 rows
    parts = [torch.arange(c, dtype=torch.float32).mul(1).add(100.0 * r)
             .reshape(c, 1, 1).expand(c, n, 2).contiguous() for r, c in enumerate(counts)]
    tls = [torch.full((n,), 10.0 + r) for r in range(3)]
    p, tl = tp.assemble(parts, tls, owner)
    assert p.shape == (5, n, 2)
    expect = torch.tensor([0.0, 100.0, 101.0, 200.0, 201.0])
    for row in range(n):
        for e in range(2):
            assert torch.equal(p[:, row, e], expect)
    # global chunk c covers vocab rows [1024 c, 1024 (c + 1)): its owner is the block holding it
    for c in range(p.shape[0]):
        r = int(p[c, 0, 0].item()) // 100
        assert sh[r][0] <= 1024 * c < sh[r][0] + sh[r][1]
    assert tl.tolist()[:4] == [10.0 + o for o in owner.tolist()[:4]]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        vocab, n = 5000, 6
        sh = tp.vocab_shards(vocab, world)
        targets = torch.tensor([0, 1023, 1024, 4999, 2047, 3000])
        owner = tp.owner_of(targets, sh)
        start, size = sh[rank]
        s_local = -(-size // 1024)
        # rank r's chunk c carries the value (global chunk index); rank r's target logit is r
        c0 = start // 1024
        local = torch.arange(c0, c0 + s_local, dtype=torch.float32).view(-1, 1, 1).expand(
            s_local, n, 2).contiguous()
        tl = torch.full((n,), float(rank))
        p, t = tp.exchange(local, tl, owner)
        out[rank] = (p[:, 0, 0].tolist(), t.tolist(), owner.tolist())
    finally:
        dist.destroy_process_group()


def test_two_rank_exchange_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    chunks, tl, owner = out[0]
    assert out[0] == out[1]
    assert chunks == [0.0, 1.0, 2.0, 3.0, 4.0]          # global chunk order
    assert tl == [float(o) for o in owner]               # from the owning rank


def _dh_worker(rank, world, port, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        local = torch.full((3, 4), float(rank + 1))
        g = tp.gather_dh_partials(local)
        out[rank] = g[:, 0, 0].tolist()
    finally:
        dist.destroy_process_group()


def test_two_rank_dh_partials_gloo():
    # every rank receives the partials stacked in rank order
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_dh_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == [1.0, 2.0]
