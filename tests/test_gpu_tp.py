"""Vocab-sharded forward emulated on one GPU ("RL-Kernel integration roadmap for
vime", linear_logp: explicit TP vocab-shard merge; "RL-Kernel Roadmap (2026)",
TP-invariant reductions): the LM head is cut into k blocks on 1024-row
boundaries, each block's partials come from rlk_linear_logp_fwd_shard, and
rlk_linear_logp_merge must give logp and lse bitwise equal to the unsharded
rlk_linear_logp_fwd for k = 2, 4, 8 (and parity with the oracle follows)."""
import numpy as np
import pytest
import torch

import rl_post_linear_gb300 as rlk
import workloads as wl
from helpers import dev, same_bits
from rl_post_linear_gb300 import tp

pytestmark = pytest.mark.gpu


def _sharded(h, w, y, m, T, parts):
    d = h.device
    n = h.shape[0]
    vocab = w.shape[0]
    shards = tp.vocab_shards(vocab, parts)
    total = rlk.rlk_linear_logp_num_partials(vocab)
    partials = torch.empty(total, n, 2, dtype=torch.float32, device=d)
    target_logit = torch.zeros(n, dtype=torch.float32, device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    for start, size in shards:
        if size == 0:
            continue
        c0 = start // tp.CHUNK
        cnt = rlk.rlk_linear_logp_num_partials(size)
        rlk.rlk_linear_logp_fwd_shard(h, w[start:start + size], y, m, start, T,
                                      partials[c0:c0 + cnt], target_logit, err)
    logp = torch.empty(n, dtype=torch.float32, device=d)
    lse = torch.empty(n, dtype=torch.float32, device=d)
    rlk.rlk_linear_logp_merge(partials, total, target_logit, y, m, vocab, T, logp, lse, err)
    torch.cuda.synchronize()
    return logp, lse, int(err.item())


@pytest.mark.parametrize("n,h,vocab,T", [(256, 4096, 151936, 0.7), (300, 256, 5000, 1.0),
                                         (129, 128, 1000, 0.5)])
def test_tp_bitwise_equals_unsharded(n, h, vocab, T):
    d = dev()
    seed = n + vocab
    hid = wl.normal_bf16((n, h), seed, wl.S_HIDDEN).to(d)
    w = wl.normal_bf16((vocab, h), seed, wl.S_WEIGHT, std=0.02).to(d)
    y = wl.uniform_targets(n, vocab, seed).to(d)
    m = torch.from_numpy((np.random.default_rng(seed).random(n) < 0.9).astype(np.uint8)).to(d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    ref, ref_lse = rlk.linear_logp_fwd(hid, w, y, m, T, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for parts in (1, 2, 4, 8):
        logp, lse, e = _sharded(hid, w, y, m, T, parts)
        assert e == 0
        assert same_bits(logp.cpu(), ref.cpu()) and same_bits(lse.cpu(), ref_lse.cpu()), parts


def test_tp_flags_out_of_range_targets_and_rejects_unaligned_blocks():
    d = dev()
    n, h, vocab = 64, 128, 3000
    hid = wl.normal_bf16((n, h), 1, wl.S_HIDDEN).to(d)
    w = wl.normal_bf16((vocab, h), 1, wl.S_WEIGHT, std=0.02).to(d)
    y = wl.uniform_targets(n, vocab, 1)
    y[5] = vocab + 3
    y = y.to(d)
    logp, _, e = _sharded(hid, w, y, None, 1.0, 3)
    assert e & rlk.RLK_DEVERR_TARGET_RANGE and torch.isnan(logp[5]).item()
    part = torch.empty(4, n, 2, dtype=torch.float32, device=d)
    tl = torch.empty(n, dtype=torch.float32, device=d)
    with pytest.raises(rlk.RlkError) as ex:
        rlk.rlk_linear_logp_fwd_shard(hid, w[100:1100], y, None, 100, 1.0, part, tl)
    assert ex.value.status == rlk.RLK_ERR_UNSUPPORTED
