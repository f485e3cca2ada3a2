"""Tensor-parallel (vocab-sharded) forward and backward on top of the shard / merge
entry points.

"RL-Kernel integration roadmap for vime", linear_logp section (TP support,
with the merge of the vocabulary shards as an explicit step); "RL-Kernel
Roadmap (2026)", TP-invariant reductions.  Each rank holds a contiguous block of LM-head rows starting on a
1024-row boundary, computes its block's partials with
``rlk_linear_logp_fwd_shard``, and the ranks exchange them once: an
all-gather of the (max, sum) pairs, concatenated in rank order (which is the
global chunk order), and of the target-logit rows, each row taken from the
rank whose block holds its target.  ``rlk_linear_logp_merge`` then gives logp
and lse bitwise equal to the unsharded forward.

The backward needs one more exchange: every rank computes its block's fp32
contribution to dh with ``rlk_linear_logp_bwd_shard`` (and its own rows of dW);
``gather_dh_partials`` all-gathers the partials in rank order and
``rlk_linear_logp_dh_merge`` sums them in that order and rounds once, so every
rank gets the same dh whatever the transport.

The exchanges are the only collectives; every arithmetic step runs in the
library's kernels.
"""
from __future__ import annotations

import torch

CHUNK = 1024


def vocab_shards(vocab: int, parts: int):
    """[(start, size)] of `parts` contiguous blocks covering [0, vocab), every start a
    multiple of 1024 and every block but the last a multiple of 1024 rows (so that the
    sharded result is bitwise equal to the unsharded one).  Blocks may be empty when
    vocab is small."""
    if parts < 1 or vocab < 1:
        raise ValueError("parts and vocab must be positive")
    chunks = -(-vocab // CHUNK)
    out = []
    for i in range(parts):
        c0 = chunks * i // parts
        c1 = chunks * (i + 1) // parts
        start = min(c0 * CHUNK, vocab)
        end = min(c1 * CHUNK, vocab)
        out.append((start, end - start))
    return out


def owner_of(targets: torch.Tensor, shards):
    """Index of the block holding each target (-1 for targets outside every block)."""
    owner = torch.full_like(targets, -1)
    for i, (start, size) in enumerate(shards):
        if size > 0:
            owner[(targets >= start) & (targets < start + size)] = i
    return owner


def assemble(partials_per_rank, target_logit_per_rank, owner):
    """Concatenate per-rank partials [S_r, N, 2] in rank order and pick each row's target
    logit from its owning rank.  Pure data movement (no arithmetic on the values)."""
    partials = torch.cat([p.reshape(-1, p.shape[-2], 2) for p in partials_per_rank], dim=0)
    stacked = torch.stack(target_logit_per_rank, dim=0)
    idx = owner.clamp(min=0).unsqueeze(0)
    target_logit = torch.gather(stacked, 0, idx).squeeze(0)
    return partials.contiguous(), target_logit.contiguous()


def exchange(local_partials, local_target_logit, owner, group=None):
    """All-gather the block partials and target logits of every rank (torch.distributed),
    then assemble them; returns (partials [S, N, 2], target_logit [N])."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    sizes = [torch.zeros(1, dtype=torch.int64, device=local_partials.device) for _ in range(world)]
    dist.all_gather(sizes, torch.tensor([local_partials.shape[0]], dtype=torch.int64,
                                        device=local_partials.device), group=group)
    n = local_partials.shape[1]
    counts = [int(s.item()) for s in sizes]
    most = max(counts)
    padded = torch.zeros(most, n, 2, dtype=local_partials.dtype, device=local_partials.device)
    padded[:local_partials.shape[0]] = local_partials
    gathered = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(gathered, padded, group=group)           # equal sizes: pad, then trim
    gathered = [g[:c] for g, c in zip(gathered, counts)]
    tl = [torch.empty_like(local_target_logit) for _ in range(world)]
    dist.all_gather(tl, local_target_logit.contiguous(), group=group)
    return assemble(gathered, tl, owner)


def gather_dh_partials(local_partial, group=None):
    """All-gather every rank's fp32 dh partial [N, H]; returns [world, N, H] in rank order
    (the order rlk_linear_logp_dh_merge sums in).  Pure data movement."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    gathered = [torch.empty_like(local_partial) for _ in range(world)]
    dist.all_gather(gathered, local_partial.contiguous(), group=group)
    return torch.stack(gathered, dim=0)
