"""Data-parallel exchange of the LM-head weight gradient, in a fixed rank order.

"RL-Kernel Roadmap (2026)", WS2: a deterministic all-reduce sums the ranks'
contributions in a fixed order with fp32 accumulation.  With the batch's tokens
split over data-parallel ranks, each rank's backward
(``rlk_linear_logp_bwd_dw_partial``) leaves an unrounded fp32 partial of dW
[V, H]; dhidden needs no exchange (a token's row depends on that token alone).

The exchange here is a reduce-scatter made deterministic, then an all-gather:

1. ``dw_row_blocks`` cuts the V rows into one contiguous block per rank.
2. ``reduce_scatter_dw``: one all-to-all sends block b of every rank's partial
   to rank b, which receives the world's partials of its block stacked in rank
   order and sums them with ``rlk_linear_logp_dw_merge`` (fp32, rank 0 first,
   one bf16 rounding).  The bytes moved per rank are those of a ring
   reduce-scatter; the order of the sum is the rank order whatever the
   transport does.
3. ``all_gather_dw`` gathers the bf16 blocks into the whole dW on every rank
   (a sharded optimiser can keep its block instead).

The merged dW therefore depends only on the partials and the number of ranks,
never on the collective's algorithm or timing.
"""
from __future__ import annotations

import torch


def dw_row_blocks(vocab: int, world: int):
    """[(start, rows)] per rank: contiguous blocks of the V rows, the first
    ``vocab % world`` blocks one row longer."""
    if world < 1 or vocab < 0:
        raise ValueError("world must be >= 1 and vocab >= 0")
    base, extra = divmod(vocab, world)
    out, start = [], 0
    for r in range(world):
        rows = base + (1 if r < extra else 0)
        out.append((start, rows))
        start += rows
    return out


def _default_merge(stacked: torch.Tensor) -> torch.Tensor:
    import rl_post_linear_gb300 as rlk
    out = torch.empty(stacked.shape[1:], dtype=torch.bfloat16, device=stacked.device)
    rlk.rlk_linear_logp_dw_merge(stacked, out)
    return out


def reduce_scatter_dw(dw_partial: torch.Tensor, group=None, merge=None):
    """This rank's block of dW = bf16(sum over ranks, in rank order, of their fp32
    partials).  Returns (block [rows, H] bf16, (start, rows)).

    ``merge`` maps the received partials [world, rows, H] (rank order) to the
    block; the default is ``rlk_linear_logp_dw_merge``."""
    import torch.distributed as dist
    if dw_partial.dtype != torch.float32 or dw_partial.dim() != 2 or not dw_partial.is_contiguous():
        raise ValueError("dw_partial must be a contiguous [V, H] float32 tensor")
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    v, h = dw_partial.shape
    blocks = dw_row_blocks(v, world)
    start, rows = blocks[rank]
    recv = torch.empty(world * rows, h, dtype=dw_partial.dtype, device=dw_partial.device)
    dist.all_to_all_single(recv, dw_partial, output_split_sizes=[rows] * world,
                           input_split_sizes=[n for _, n in blocks], group=group)
    stacked = recv.view(world, rows, h)
    block = (merge or _default_merge)(stacked)
    return block, (start, rows)


def all_gather_dw(block: torch.Tensor, vocab: int, group=None) -> torch.Tensor:
    """The whole dW [V, H] from every rank's block (rank order = row order)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    blocks = dw_row_blocks(vocab, world)
    most = max(n for _, n in blocks)
    h = block.shape[1]
    padded = torch.zeros(most, h, dtype=block.dtype, device=block.device)
    padded[:block.shape[0]] = block
    gathered = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(gathered, padded, group=group)        # equal sizes: pad, then trim
    return torch.cat([g[:n] for g, (_, n) in zip(gathered, blocks)], dim=0)
