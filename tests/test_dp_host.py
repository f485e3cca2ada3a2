"""Host logic of the data-parallel dW exchange, on CPU over gloo: the row
blocks, the all-to-all that hands each rank the world's partials of its block
in rank order, and the all-gather of the merged blocks.  The GPU merge is
replaced here by a plain sequential fp32 sum, so the test checks what the
exchange delivers and in which order ("RL-Kernel Roadmap (2026)", WS2:
deterministic all-reduce in a fixed rank order)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

from rl_post_linear_gb300 import dp


@pytest.mark.parametrize("vocab,world", [(151936, 1), (151936, 2), (151936, 8), (129280, 3),
                                         (5, 8), (0, 2), (7, 7)])
def test_row_blocks(vocab, world):
    b = dp.dw_row_blocks(vocab, world)
    assert len(b) == world
    pos = 0
    for start, rows in b:
        assert start == pos and rows >= 0
        pos += rows
    assert pos == vocab
    sizes = [n for _, n in b]
    assert max(sizes) - min(sizes) <= 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _partial(rank, vocab, h):
    # rank r's partial: row v, column c holds 1000 r + v + c / 100; row 0 of every rank also
    # carries a term whose fp32 sum depends on the order: 1e8, 1, -1e8, 0, ... by rank
    p = (torch.arange(vocab, dtype=torch.float32).unsqueeze(1) + 1000.0 * rank
         + torch.arange(h, dtype=torch.float32).unsqueeze(0) / 100)
    p[0, 0] = [1e8, 1.0, -1e8][rank] if rank < 3 else 0.0
    return p.contiguous()


def _seq_merge(stacked):
    out = stacked[0].clone()
    for r in range(1, stacked.shape[0]):
        out = out + stacked[r]
    return out


def _worker(rank, world, port, vocab, h, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seen = {}

        def merge(stacked):
            seen["stacked"] = stacked.clone()
            return _seq_merge(stacked)

        block, (start, rows) = dp.reduce_scatter_dw(_partial(rank, vocab, h), merge=merge)
        full = dp.all_gather_dw(block, vocab)
        out[rank] = (seen["stacked"], block, start, rows, full)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,vocab", [(2, 7), (3, 10)])
def test_reduce_scatter_and_gather(world, vocab):
    h = 4
    mgr = mp.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.spawn(_worker, args=(world, port, vocab, h, out), nprocs=world, join=True)
    partials = [_partial(r, vocab, h) for r in range(world)]
    expect_full = _seq_merge(torch.stack(partials))
    blocks = dp.dw_row_blocks(vocab, world)
    for rank in range(world):
        stacked, block, start, rows, full = out[rank]
        assert (start, rows) == blocks[rank]
        # the world's partials of this rank's block, in rank order
        for r in range(world):
            assert torch.equal(stacked[r], partials[r][start:start + rows])
        assert torch.equal(block, expect_full[start:start + rows])
        assert torch.equal(full, expect_full)
    # the order-sensitive entry: 1e8 + 1 rounds to 1e8 in fp32 (its spacing there is 8), so in
    # rank order (1e8 + 1) - 1e8 is 0, where 1e8 + (1 - 1e8) would be 8 and (1e8 - 1e8) + 1 is 1
    assert expect_full[0, 0].item() == (0.0 if world >= 3 else 1e8)
