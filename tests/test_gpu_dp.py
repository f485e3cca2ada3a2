"""Data-parallel backward of the LM head ("RL-Kernel Roadmap (2026)", WS2:
deterministic all-reduce, fixed rank order with fp32 accumulation): a batch
split over k emulated ranks, each rank's rlk_linear_logp_bwd_dw_partial
leaving an unrounded fp32 dW partial, merged by rlk_linear_logp_dw_merge in
rank order.  The merged dW is within the 2e-3 gradient contract of the fp64
oracle's dW for the whole batch and bitwise reproducible; each rank's dhidden
rows are bitwise the whole batch's (per-token gradients need no exchange); a
single partial rounds to rlk_linear_logp_bwd's dW bit for bit; and the merge
equals a sequential fp32 sum in rank order, rounded once."""
import numpy as np
import pytest
import torch

import oracle
import rl_post_linear_gb300 as rlk
import workloads as wl
from helpers import GRAD_REL_L2, dev, f64, rel_l2, same_bits

pytestmark = pytest.mark.gpu


def _case(n, h, v, seed):
    hidden = wl.normal_bf16((n, h), seed, wl.S_HIDDEN)
    weight = wl.normal_bf16((v, h), seed, wl.S_WEIGHT, std=0.2)
    targets = wl.uniform_targets(n, v, seed)
    rng = np.random.default_rng(seed)
    mask = torch.from_numpy((rng.random(n) < 0.8).astype(np.uint8))
    g = rng.standard_normal(n) / n
    g[mask.numpy() == 0] = 0.0
    return hidden, weight, targets, mask, g


def _rank_partials(hd, wd, yd, md, gd, lse, T, splits):
    n, h = hd.shape
    v = wd.shape[0]
    parts = torch.empty(len(splits) - 1, v, h, dtype=torch.float32, device=hd.device)
    dh = torch.empty_like(hd)
    for r in range(len(splits) - 1):
        a, b = splits[r], splits[r + 1]
        ws = torch.empty(rlk.rlk_linear_logp_bwd_workspace_bytes(b - a, h, v), dtype=torch.uint8,
                         device=hd.device)
        dh_r = torch.empty(b - a, h, dtype=torch.bfloat16, device=hd.device)
        rlk.rlk_linear_logp_bwd_dw_partial(hd[a:b], wd, yd[a:b], md[a:b], gd[a:b], lse[a:b], T,
                                           dh_r, parts[r], ws)
        dh[a:b] = dh_r
    return parts, dh


@pytest.mark.parametrize("n,h,v,T,splits", [(600, 256, 40000, 0.8, [0, 200, 350, 600]),
                                            (300, 128, 3000, 1.0, [0, 1, 150, 299, 300])])
def test_dp_partials_merged_in_rank_order(n, h, v, T, splits):
    hidden, weight, targets, mask, g = _case(n, h, v, n + v)
    d = dev()
    hd, wd, yd, md = hidden.to(d), weight.to(d), targets.to(d), mask.to(d)
    gd = torch.tensor(g, dtype=torch.float32, device=d)
    _, lse = rlk.linear_logp_fwd(hd, wd, yd, md, T)
    parts, dh = _rank_partials(hd, wd, yd, md, gd, lse, T, splits)
    dw = torch.empty_like(wd)
    rlk.rlk_linear_logp_dw_merge(parts, dw)
    # bitwise reproducible
    parts2, dh2 = _rank_partials(hd, wd, yd, md, gd, lse, T, splits)
    dw2 = torch.empty_like(wd)
    rlk.rlk_linear_logp_dw_merge(parts2, dw2)
    torch.cuda.synchronize()
    assert same_bits(parts.cpu(), parts2.cpu()) and same_bits(dw.cpu(), dw2.cpu())
    # the merge is the sequential fp32 sum in rank order, rounded once (RNE)
    acc = parts[0].clone()
    for r in range(1, parts.shape[0]):
        acc = acc + parts[r]
    assert same_bits(dw.cpu(), acc.to(torch.bfloat16).cpu())
    # per-token rows need no exchange: bitwise the whole batch's
    dh_full, dw_full = rlk.linear_logp_bwd(hd, wd, yd, md, gd, lse, T)
    assert same_bits(dh.cpu(), dh_full.cpu())
    # against the fp64 oracle's gradient of the whole batch
    h64, w64 = f64(hidden), f64(weight)
    _, lse_o = oracle.linear_logp_fwd_parallel(h64, w64, targets.numpy(), mask.numpy(), T)
    g32 = gd.cpu().double().numpy()
    dw_o = oracle.linear_logp_bwd_dw_parallel(h64, w64, targets.numpy(), mask.numpy(), g32, lse_o,
                                              T, 0, v)
    e_dw = rel_l2(dw.cpu(), dw_o)
    e_full = rel_l2(dw_full.cpu(), dw_o)
    print("dp k=%d n=%d v=%d: merged dW rel-L2 %.3e (single-rank dW %.3e)"
          % (len(splits) - 1, n, v, e_dw, e_full))
    assert e_dw <= GRAD_REL_L2


def test_single_partial_rounds_to_the_unsplit_backward():
    hidden, weight, targets, mask, g = _case(257, 192, 2000, 5)
    d = dev()
    hd, wd, yd, md = hidden.to(d), weight.to(d), targets.to(d), mask.to(d)
    gd = torch.tensor(g, dtype=torch.float32, device=d)
    _, lse = rlk.linear_logp_fwd(hd, wd, yd, md, 0.9)
    parts, dh = _rank_partials(hd, wd, yd, md, gd, lse, 0.9, [0, 257])
    dw = torch.empty_like(wd)
    rlk.rlk_linear_logp_dw_merge(parts, dw)
    dh1, dw1 = rlk.linear_logp_bwd(hd, wd, yd, md, gd, lse, 0.9)
    torch.cuda.synchronize()
    assert same_bits(dw.cpu(), dw1.cpu()) and same_bits(dh.cpu(), dh1.cpu())


def test_merge_argument_errors():
    lib = rlk.load()
    assert lib.rlk_linear_logp_dw_merge(None, 0, 10, 64, None, None) == rlk.RLK_ERR_INVALID_VALUE
    assert lib.rlk_linear_logp_dw_merge(None, 2, 10, 65, None, None) == rlk.RLK_ERR_UNSUPPORTED
    assert lib.rlk_linear_logp_dw_merge(None, 2, 0, 64, None, None) == rlk.RLK_OK
    assert lib.rlk_linear_logp_dw_merge(None, 2, 10, 64, None, None) == rlk.RLK_ERR_INVALID_VALUE
