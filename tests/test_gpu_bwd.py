"""GPU backward vs the fp64 oracle: dh and dW relative L2 <= 2e-3, exact zeros
on inactive rows, dh batch invariance and dW run-to-run determinism.

Chunked-recompute backward ("RL-Kernel Roadmap (2026)", P0.2;
"RL-Kernel integration roadmap for vime", linear_logp).
"""
import numpy as np
import pytest
import torch

import oracle
import rl_post_linear_gb300 as rlk
import workloads as wl
from helpers import GRAD_REL_L2, dev, f64, rel_l2, same_bits

pytestmark = pytest.mark.gpu


def _case(n, h, v, seed, std=0.05, active=0.85):
    hidden = wl.normal_bf16((n, h), seed, wl.S_HIDDEN)
    weight = wl.normal_bf16((v, h), seed, wl.S_WEIGHT, std=std)
    targets = wl.uniform_targets(n, v, seed)
    g = np.random.default_rng(seed)
    mask = torch.from_numpy((g.random(n) < active).astype(np.uint8))
    grad = g.standard_normal(n) / max(1, n)
    grad[mask.numpy() == 0] = 0.0
    return hidden, weight, targets, mask, grad


def _gpu(hidden, weight, targets, mask, grad, T):
    d = dev()
    h, w, y = hidden.to(d), weight.to(d), targets.to(d)
    m = None if mask is None else mask.to(d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    logp, lse = rlk.linear_logp_fwd(h, w, y, m, T, err)
    g = torch.tensor(grad, dtype=torch.float32, device=d)
    dh, dw = rlk.linear_logp_bwd(h, w, y, m, g, lse, T, err)
    torch.cuda.synchronize()
    return dh.cpu(), dw.cpu(), lse.cpu(), int(err.item())


def _oracle(hidden, weight, targets, mask, grad, T):
    h64, w64 = f64(hidden), f64(weight)
    m = None if mask is None else mask.numpy()
    _, lse = oracle.linear_logp_fwd_parallel(h64, w64, targets.numpy(), m, T)
    dh = oracle.linear_logp_bwd_dh_parallel(h64, w64, targets.numpy(), m, grad, lse, T)
    dw = oracle.linear_logp_bwd_dw_parallel(h64, w64, targets.numpy(), m, grad, lse, T, 0,
                                            w64.shape[0])
    return dh, dw


def test_tiny_parity():
    w = wl.tiny_fwd(0)
    g = np.random.default_rng(0).standard_normal(w.n) / w.n_active
    g[w.mask.numpy() == 0] = 0
    dh, dw, _, err = _gpu(w.hidden, w.weight, w.targets, w.mask, g, w.temperature)
    assert err == 0
    dh_o, dw_o = _oracle(w.hidden, w.weight, w.targets, w.mask, g, w.temperature)
    e_dh, e_dw = rel_l2(dh, dh_o), rel_l2(dw, dw_o)
    print("bwd parity tiny: rel-L2 dh %.3e dw %.3e" % (e_dh, e_dw))
    assert e_dh <= GRAD_REL_L2 and e_dw <= GRAD_REL_L2
    assert torch.all(dh[w.mask == 0] == 0)


@pytest.mark.parametrize("n,h,v,T", [(300, 128, 40000, 0.7), (129, 256, 1000, 1.0),
                                     (70, 64, 2 * 32768 + 300, 1.5)])
def test_multi_chunk_ragged_parity(n, h, v, T):
    hidden, weight, targets, mask, grad = _case(n, h, v, n + h + v)
    targets[5] = targets[6] = targets[40] = 17          # a vocab row hit by several tokens
    mask[5] = mask[6] = mask[40] = 1
    grad[[5, 6, 40]] = [0.02, -0.015, 0.01]             # so that the fp32 target term dominates
    dh, dw, _, err = _gpu(hidden, weight, targets, mask, grad, T)
    assert err == 0
    dh_o, dw_o = _oracle(hidden, weight, targets, mask, grad, T)
    e_dh, e_dw = rel_l2(dh, dh_o), rel_l2(dw, dw_o)
    print("bwd parity n=%d h=%d v=%d: rel-L2 dh %.3e dw %.3e" % (n, h, v, e_dh, e_dw))
    assert e_dh <= GRAD_REL_L2 and e_dw <= GRAD_REL_L2
    # the row hit by three tokens: every element within one bf16 rounding of the oracle
    # (a single 128-element row can exceed 2e-3 rel-L2 from the final rounding alone)
    row, ref = f64(dw[17]), dw_o[17]
    assert np.all(np.abs(row - ref) <= 2.0 ** -8 * np.abs(ref) * 1.001 + 2.0 ** -16 * np.abs(ref).max())
    assert torch.all(dh[mask == 0] == 0)


def test_dh_batch_invariance_and_dw_determinism():
    n, h, v = 300, 128, 5000
    hidden, weight, targets, mask, grad = _case(n, h, v, 11)
    dh, dw, _, _ = _gpu(hidden, weight, targets, mask, grad, 0.7)
    dh2, dw2, _, _ = _gpu(hidden, weight, targets, mask, grad, 0.7)
    assert same_bits(dh, dh2) and same_bits(dw, dw2)
    for a, b in ((0, 1), (0, 128), (100, 300), (17, 211)):
        dhp, _, _, _ = _gpu(hidden[a:b], weight, targets[a:b], mask[a:b], grad[a:b], 0.7)
        assert same_bits(dhp, dh[a:b]), (a, b)


def test_target_terms_across_sort_tiles():
    # More tokens than one 2048-key sort tile, a ragged last tile, every vocab row hit by
    # about a dozen tokens in different tiles, and unread invalid targets on inactive rows.
    n, h, v = 5000, 64, 300
    hidden, weight, targets, mask, grad = _case(n, h, v, 21, std=0.2, active=0.8)
    inactive = np.nonzero(mask.numpy() == 0)[0]
    targets[torch.from_numpy(inactive[::3])] = -5
    targets[torch.from_numpy(inactive[1::3])] = v + 7
    dh, dw, _, err = _gpu(hidden, weight, targets, mask, grad, 0.9)
    assert err == 0
    dh_o, dw_o = _oracle(hidden, weight, targets, mask, grad, 0.9)
    e_dh, e_dw = rel_l2(dh, dh_o), rel_l2(dw, dw_o)
    print("bwd parity n=%d v=%d (3 sort tiles): rel-L2 dh %.3e dw %.3e" % (n, v, e_dh, e_dw))
    assert e_dh <= GRAD_REL_L2 and e_dw <= GRAD_REL_L2
    # dh rows are per token: permuting the tokens permutes dh bit for bit
    perm = torch.from_numpy(np.random.default_rng(1).permutation(n))
    dhp, _, _, _ = _gpu(hidden[perm], weight, targets[perm], mask[perm], grad[perm.numpy()], 0.9)
    assert same_bits(dhp, dh[perm])


def _bwd_raw(hidden, weight, targets, mask, grad, T, fill=0xFF):
    """The C-ABI backward with outputs and workspace pre-filled with NaN bytes, so that
    a row or tile nobody writes (or a stale workspace row that gets read) shows."""
    d = dev()
    h, w, y = hidden.to(d), weight.to(d), targets.to(d)
    m = None if mask is None else mask.to(d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    _, lse = rlk.linear_logp_fwd(h, w, y, m, T, err)
    g = torch.tensor(grad, dtype=torch.float32, device=d)
    n, hd = hidden.shape
    dh = torch.empty_like(h).view(torch.uint8).fill_(fill).view(torch.bfloat16)
    dw = torch.empty_like(w).view(torch.uint8).fill_(fill).view(torch.bfloat16)
    ws = torch.full((rlk.rlk_linear_logp_bwd_workspace_bytes(n, hd, w.shape[0]),), fill,
                    dtype=torch.uint8, device=d)
    rlk.rlk_linear_logp_bwd(h, w, y, m, g, lse, T, dh, dw, ws, err)
    torch.cuda.synchronize()
    return dh.cpu(), dw.cpu(), int(err.item())


@pytest.mark.parametrize("n,active", [(700, 0.3), (333, 0.9), (2100, 0.05)])
def test_masked_batch_equals_its_packed_active_rows(n, active):
    # The backward runs its GEMMs over the active rows only, gathered in ascending token
    # order: a masked batch gives, bit for bit, the dh rows and the dW of the batch made
    # of its active rows alone, and zero dh rows for the rest.
    h, v = 128, 40000                      # two vocabulary chunks, a ragged one last
    hidden, weight, targets, mask, grad = _case(n, h, v, 31 + n, std=0.1, active=active)
    dh, dw, err = _bwd_raw(hidden, weight, targets, mask, grad, 0.8)
    assert err == 0
    act = torch.from_numpy(np.nonzero(mask.numpy())[0])
    dhp, dwp, errp = _bwd_raw(hidden[act], weight, targets[act], None, grad[act.numpy()], 0.8)
    assert errp == 0
    assert same_bits(dh[act], dhp)
    assert same_bits(dw, dwp)
    assert torch.all(dh[mask == 0].float() == 0)
    dh_o, dw_o = _oracle(hidden, weight, targets, mask, grad, 0.8)
    assert rel_l2(dh, dh_o) <= GRAD_REL_L2 and rel_l2(dw, dw_o) <= GRAD_REL_L2
    # the inactive rows are never read: NaN padding changes nothing
    nan_pad = hidden.clone()
    nan_pad[mask == 0] = float("nan")
    dhn, dwn, errn = _bwd_raw(nan_pad, weight, targets, mask, grad, 0.8)
    assert errn == 0 and same_bits(dhn, dh) and same_bits(dwn, dw)


def test_all_masked_batch_gives_zero_gradients():
    n, h, v = 300, 128, 5000
    hidden, weight, targets, mask, grad = _case(n, h, v, 41)
    mask.zero_()
    grad[:] = 0.0
    dh, dw, err = _bwd_raw(hidden, weight, targets, mask, grad, 1.0)
    assert err == 0
    assert torch.all(dh.float() == 0) and torch.all(dw.float() == 0)
    # one active row
    mask[177] = 1
    grad[177] = 0.5
    dh, dw, err = _bwd_raw(hidden, weight, targets, mask, grad, 1.0)
    assert err == 0
    assert torch.all(dh[mask == 0].float() == 0)
    dh_o, dw_o = _oracle(hidden, weight, targets, mask, grad, 1.0)
    assert rel_l2(dh, dh_o) <= GRAD_REL_L2 and rel_l2(dw, dw_o) <= GRAD_REL_L2


def _dominant_case(n, h, v, seed, rows_by_chunk):
    """Random head plus, for the listed rows, one planted class per row in the given chunk
    whose logit is about 17 (p > 0.9 at T = 1): a dominant non-target class."""
    hidden, weight, targets, mask, grad = _case(n, h, v, seed, std=0.02, active=1.0)
    rng = np.random.default_rng(seed + 100)
    w = weight.float()
    hf = hidden.float()
    for chunk, rows in rows_by_chunk.items():
        lo, hi = chunk * 32768, min(v, (chunk + 1) * 32768)
        for t in rows:
            a = int(rng.integers(lo, hi))
            w[a] += 2.2 * hf[t] / hf[t].norm()
    return hidden, w.to(torch.bfloat16), targets, mask, grad


def test_dominant_classes_in_some_chunks_and_a_reused_workspace():
    # Three vocabulary chunks: rows 0-39 have a dominant class in chunk 0, rows 40-79 in
    # chunk 2, none in chunk 1 (whose dominant-class sort is skipped).  Then a head with no
    # dominant class at all through the same workspace: the lists left by the first call
    # must not be read.
    n, h, v, T = 200, 64, 70000, 1.0
    hidden, weight, targets, mask, grad = _dominant_case(
        n, h, v, 51, {0: range(0, 40), 2: range(40, 80)})
    d = dev()
    ws = torch.empty(rlk.rlk_linear_logp_bwd_workspace_bytes(n, h, v), dtype=torch.uint8,
                     device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)

    def run(hid, wt):
        hd, wd, yd, md = hid.to(d), wt.to(d), targets.to(d), mask.to(d)
        _, lse = rlk.linear_logp_fwd(hd, wd, yd, md, T, err)
        g = torch.tensor(grad, dtype=torch.float32, device=d)
        dh, dw = torch.empty_like(hd), torch.empty_like(wd)
        rlk.rlk_linear_logp_bwd(hd, wd, yd, md, g, lse, T, dh, dw, ws, err)
        torch.cuda.synchronize()
        return dh.cpu(), dw.cpu(), lse.cpu()

    dh, dw, lse = run(hidden, weight)
    assert int(err.item()) == 0
    p_max = float(torch.exp(hidden.float() @ weight.float().t() / T
                            - lse[:, None]).max(dim=1).values[:80].min())
    assert p_max > 0.6                                  # the planted classes dominate
    dh_o, dw_o = _oracle(hidden, weight, targets, mask, grad, T)
    e_dh, e_dw = rel_l2(dh, dh_o), rel_l2(dw, dw_o)
    print("dominant classes in chunks 0 and 2: rel-L2 dh %.3e dw %.3e" % (e_dh, e_dw))
    assert e_dh <= GRAD_REL_L2 and e_dw <= GRAD_REL_L2
    plain = wl.normal_bf16((v, h), 52, wl.S_WEIGHT, std=0.02)
    dh2, dw2, _ = run(hidden, plain)
    assert int(err.item()) == 0
    dh2_o, dw2_o = _oracle(hidden, plain, targets, mask, grad, T)
    assert rel_l2(dh2, dh2_o) <= GRAD_REL_L2 and rel_l2(dw2, dw2_o) <= GRAD_REL_L2


def test_single_class_vocabulary_gives_zero_up_to_lse_rounding():
    # V = 1: p = 1 for every row, so the exact gradient g (delta - p) / T is 0.  The kernels
    # rebuild log2 p as S k - lse log2(e) from the forward's fp32 lse, which is off by about
    # one fp32 ulp of lse: the target entry's coefficient (g / T)(1 - p) is then of order
    # 2^-23 |g| / T instead of 0.  The outputs must stay at that rounding level.
    T = 0.9
    for n in (1, 5, 300):
        hidden, weight, targets, mask, grad = _case(n, 64, 1, 61 + n, std=0.3, active=0.8)
        dh, dw, err = _bwd_raw(hidden, weight, targets, mask, grad, T)
        assert err == 0
        assert torch.all(dh[mask == 0].float() == 0)
        lse_scale = float((hidden.float() @ weight.float().t()).abs().max()) / T + 1.0
        g_max = float(np.abs(grad).max()) / T
        bound_dh = 8 * 2.0 ** -23 * lse_scale * g_max * float(weight.float().abs().max())
        bound_dw = 8 * 2.0 ** -23 * lse_scale * g_max * float(hidden.float().abs().max()) * n
        assert float(dh.float().abs().max()) <= bound_dh
        assert float(dw.float().abs().max()) <= bound_dw


@pytest.mark.parametrize("n,h,v", [(1, 64, 3), (40, 64, 2), (3, 192, 7)])
def test_tiny_vocabulary_and_batch(n, h, v):
    hidden, weight, targets, mask, grad = _case(n, h, v, 71 + n * v, std=0.2, active=1.0)
    dh, dw, err = _bwd_raw(hidden, weight, targets, mask, grad, 0.8)
    assert err == 0
    dh_o, dw_o = _oracle(hidden, weight, targets, mask, grad, 0.8)
    e_dh, e_dw = rel_l2(dh, dh_o), rel_l2(dw, dw_o)
    print("bwd n=%d h=%d v=%d: rel-L2 dh %.3e dw %.3e" % (n, h, v, e_dh, e_dw))
    assert e_dh <= GRAD_REL_L2 and e_dw <= GRAD_REL_L2
