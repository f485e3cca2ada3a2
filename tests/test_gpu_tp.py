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


def _sharded_bwd(h, w, y, m, g, lse, T, bounds):
    """Backward over the vocab blocks [bounds[i], bounds[i+1]), then the dh merge."""
    d = h.device
    n, hdim = h.shape
    vocab = w.shape[0]
    parts = len(bounds) - 1
    partials = torch.empty(parts, n, hdim, dtype=torch.float32, device=d)
    dw = torch.empty_like(w)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    for r in range(parts):
        a, b = bounds[r], bounds[r + 1]
        ws = torch.empty(max(256, rlk.rlk_linear_logp_bwd_workspace_bytes(n, hdim, b - a)),
                         dtype=torch.uint8, device=d)
        rlk.rlk_linear_logp_bwd_shard(h, w[a:b], y, m, g, lse, a, vocab, T, partials[r],
                                      dw[a:b], ws, err)
    dh = torch.empty_like(h)
    rlk.rlk_linear_logp_dh_merge(partials, dh)
    torch.cuda.synchronize()
    return dh, dw, int(err.item())


@pytest.mark.parametrize("n,h,vocab,T,std", [(200, 256, 70000, 0.8, 0.05),
                                             (150, 128, 9000, 0.3, 0.5)])
def test_tp_backward(n, h, vocab, T, std):
    # dW blocks are bitwise the rows of the unsharded dW (a row's arithmetic does not depend
    # on the blocking); one block reproduces the unsharded dh bit for bit; more blocks change
    # only the fp32 order in which dh's vocabulary sum is taken.
    d = dev()
    seed = n + vocab
    hid = wl.normal_bf16((n, h), seed, wl.S_HIDDEN).to(d)
    w = wl.normal_bf16((vocab, h), seed, wl.S_WEIGHT, std=std).to(d)
    y = wl.uniform_targets(n, vocab, seed).to(d)
    m = torch.from_numpy((np.random.default_rng(seed).random(n) < 0.9).astype(np.uint8)).to(d)
    g = torch.tensor(np.random.default_rng(seed + 1).standard_normal(n) / n, dtype=torch.float32,
                     device=d)
    _, lse = rlk.linear_logp_fwd(hid, w, y, m, T)
    dh_ref, dw_ref = rlk.linear_logp_bwd(hid, w, y, m, g, lse, T)
    dh1, dw1, e = _sharded_bwd(hid, w, y, m, g, lse, T, [0, vocab])
    assert e == 0 and same_bits(dh1.cpu(), dh_ref.cpu()) and same_bits(dw1.cpu(), dw_ref.cpu())
    import oracle
    from helpers import GRAD_REL_L2, f64, rel_l2
    h64, w64 = f64(hid.cpu()), f64(w.cpu())
    _, lse_o = oracle.linear_logp_fwd_parallel(h64, w64, y.cpu().numpy(), m.cpu().numpy(), T)
    g64 = g.cpu().double().numpy()
    dh_o = oracle.linear_logp_bwd_dh_parallel(h64, w64, y.cpu().numpy(), m.cpu().numpy(), g64,
                                              lse_o, T)
    for parts in (2, 4, 8):
        bounds = [a for a, _ in tp.vocab_shards(vocab, parts)] + [vocab]
        bounds = sorted(set(bounds))
        dhp, dwp, e = _sharded_bwd(hid, w, y, m, g, lse, T, bounds)
        assert e == 0 and same_bits(dwp.cpu(), dw_ref.cpu()), parts
        err = rel_l2(dhp.cpu(), dh_o)
        print("tp bwd parts=%d: dh rel-L2 %.3e (unsharded %.3e)" % (parts, err,
                                                                   rel_l2(dh_ref.cpu(), dh_o)))
        assert err <= GRAD_REL_L2
    # block boundaries need no alignment for the backward
    dhq, dwq, _ = _sharded_bwd(hid, w, y, m, g, lse, T, [0, 1000, vocab // 2 + 7, vocab])
    assert same_bits(dwq.cpu(), dw_ref.cpu()) and rel_l2(dhq.cpu(), dh_o) <= GRAD_REL_L2
