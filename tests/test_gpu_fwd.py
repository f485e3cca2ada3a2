"""GPU forward vs the fp64 oracle, exact identities and small invariance checks.

Forward of the fused linear selected-token log-prob ("RL-Kernel Roadmap
(2026)", P0.2; "RL-Kernel integration roadmap for vime", linear_logp).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import rl_post_linear_gb300 as rlk
import workloads as wl
from helpers import LOGP_ATOL, dev, f64, same_bits

pytestmark = pytest.mark.gpu


def _run(hidden, weight, targets, mask, T):
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    logp, lse = rlk.linear_logp_fwd(hidden.to(dev()), weight.to(dev()), targets.to(dev()),
                                    None if mask is None else mask.to(dev()), T, err)
    torch.cuda.synchronize()
    return logp.cpu(), lse.cpu(), int(err.item())


def _oracle(hidden, weight, targets, mask, T):
    return oracle.linear_logp_fwd_parallel(f64(hidden), f64(weight), targets.numpy(),
                                           None if mask is None else mask.numpy(), T)


def _compare(logp, lse, lp_o, lse_o, mask):
    act = np.ones(len(lp_o), bool) if mask is None else mask.numpy() > 0
    d = np.abs(logp.double().numpy() - lp_o)[act]
    assert d.max() <= LOGP_ATOL, d.max()
    dl = np.abs(lse.double().numpy() - lse_o)[act]
    assert dl.max() <= LOGP_ATOL, dl.max()
    if (~act).any():
        assert np.all(logp.numpy()[~act] == 0.0) and np.all(lse.numpy()[~act] == 0.0)
    return d.max()


def test_tiny_parity():
    w = wl.tiny_fwd(0)
    logp, lse, err = _run(w.hidden, w.weight, w.targets, w.mask, w.temperature)
    assert err == 0
    lp_o, lse_o = _oracle(w.hidden, w.weight, w.targets, w.mask, w.temperature)
    worst = _compare(logp, lse, lp_o, lse_o, w.mask)
    assert worst < 1e-4            # fp32 accumulation over H = 128 is far inside the bound


@pytest.mark.parametrize("n,h,v,T", [(300, 256, 5000, 0.7), (129, 64, 257, 1.3),
                                     (1, 128, 1, 1.0), (517, 192, 4097, 0.5)])
def test_ragged_multi_tile_parity(n, h, v, T):
    seed = n + v
    hidden = wl.normal_bf16((n, h), seed, wl.S_HIDDEN)
    weight = wl.normal_bf16((v, h), seed, wl.S_WEIGHT, std=0.05)
    targets = wl.uniform_targets(n, v, seed)
    g = np.random.default_rng(seed)
    mask = torch.from_numpy((g.random(n) < 0.9).astype(np.uint8))
    hidden[mask == 0] = float("nan")          # NaN padding never leaks into active rows
    logp, lse, err = _run(hidden, weight, targets, mask, T)
    assert err == 0
    lp_o, lse_o = _oracle(hidden, weight, targets, mask, T)
    worst = _compare(logp, lse, lp_o, lse_o, mask)
    print("fwd parity n=%d h=%d v=%d T=%g: max |dlogp| %.3e" % (n, h, v, T, worst))


def test_zero_weight_is_exact_and_row_independent():
    n, h, v = 200, 128, 3000
    hidden = wl.normal_bf16((n, h), 1, wl.S_HIDDEN)
    weight = torch.zeros(v, h, dtype=torch.bfloat16)
    targets = wl.uniform_targets(n, v, 1)
    logp, lse, err = _run(hidden, weight, targets, None, 0.7)
    assert err == 0
    assert torch.all(logp == logp[0]) and torch.all(lse == lse[0])
    assert abs(float(logp[0]) + math.log(v)) < 1e-5
    assert abs(float(lse[0]) - math.log(v)) < 1e-5


def test_power_of_two_temperature_is_bitwise_scaling():
    n, h, v = 150, 128, 2000
    hidden = wl.normal_bf16((n, h), 2, wl.S_HIDDEN)
    weight = wl.normal_bf16((v, h), 2, wl.S_WEIGHT, std=0.1)
    targets = wl.uniform_targets(n, v, 2)
    a, la, _ = _run(hidden, weight, targets, None, 2.0)
    b, lb, _ = _run(hidden, (weight.float() * 0.5).to(torch.bfloat16), targets, None, 1.0)
    assert same_bits(a, b) and same_bits(la, lb)


def test_duplicate_rows_and_batch_invariance():
    n, h, v = 260, 256, 3000
    hidden = wl.normal_bf16((n, h), 3, wl.S_HIDDEN)
    weight = wl.normal_bf16((v, h), 3, wl.S_WEIGHT, std=0.05)
    targets = wl.uniform_targets(n, v, 3)
    hidden[200] = hidden[5]
    targets[200] = targets[5]
    full, lfull, _ = _run(hidden, weight, targets, None, 0.7)
    assert full[200] == full[5] and lfull[200] == lfull[5]
    for a, b in ((0, 1), (5, 6), (100, 231), (250, 260), (37, 201)):
        part, lpart, _ = _run(hidden[a:b], weight, targets[a:b], None, 0.7)
        assert same_bits(part, full[a:b]) and same_bits(lpart, lfull[a:b])
    perm = torch.from_numpy(np.random.default_rng(0).permutation(n))
    p, lp, _ = _run(hidden[perm], weight, targets[perm], None, 0.7)
    assert same_bits(p, full[perm]) and same_bits(lp, lfull[perm])


def test_masked_rows_compacted_without_changing_bits():
    # A masked batch runs the GEMM over its active rows only, gathered in token order; a
    # row's result must not depend on that, nor on how many rows are active.
    n, h, v = 700, 256, 5000
    hidden = wl.normal_bf16((n, h), 6, wl.S_HIDDEN)
    weight = wl.normal_bf16((v, h), 6, wl.S_WEIGHT, std=0.05)
    targets = wl.uniform_targets(n, v, 6)
    full, lfull, _ = _run(hidden, weight, targets, None, 0.9)
    ones, lones, err = _run(hidden, weight, targets, torch.ones(n, dtype=torch.uint8), 0.9)
    assert err == 0 and same_bits(ones, full) and same_bits(lones, lfull)
    for density in (0.03, 0.5, 0.97):
        mask = torch.from_numpy((np.random.default_rng(int(density * 100)).random(n) < density)
                                .astype(np.uint8))
        part, lpart, err = _run(hidden, weight, targets, mask, 0.9)
        act = mask > 0
        assert err == 0 and same_bits(part[act], full[act]) and same_bits(lpart[act], lfull[act])
        assert torch.all(part[~act] == 0) and torch.all(lpart[~act] == 0)
    last = torch.zeros(n, dtype=torch.uint8)
    last[n - 1] = 1
    one, lone, _ = _run(hidden, weight, targets, last, 0.9)
    assert same_bits(one[n - 1:], full[n - 1:]) and torch.all(one[:n - 1] == 0)
    none, lnone, err = _run(hidden, weight, targets, torch.zeros(n, dtype=torch.uint8), 0.9)
    assert err == 0 and torch.all(none == 0) and torch.all(lnone == 0)


def test_invalid_targets_flagged_and_inactive_targets_unread():
    n, h, v = 40, 64, 500
    hidden = wl.normal_bf16((n, h), 4, wl.S_HIDDEN)
    weight = wl.normal_bf16((v, h), 4, wl.S_WEIGHT, std=0.05)
    targets = wl.uniform_targets(n, v, 4)
    mask = torch.ones(n, dtype=torch.uint8)
    mask[3] = 0
    targets[3] = -77                       # inactive: never read, no flag
    logp, _, err = _run(hidden, weight, targets, mask, 1.0)
    assert err == 0 and float(logp[3]) == 0.0
    targets[7] = v
    targets[9] = -1
    logp, _, err = _run(hidden, weight, targets, mask, 1.0)
    assert err & rlk.RLK_DEVERR_TARGET_RANGE
    assert math.isnan(float(logp[7])) and math.isnan(float(logp[9]))
    assert np.isfinite(logp.numpy()[[0, 1, 2, 4, 5, 6, 8, 10]]).all()


def test_empty_batch_is_a_noop():
    weight = torch.zeros(10, 64, dtype=torch.bfloat16, device=dev())
    logp, lse = rlk.linear_logp_fwd(torch.zeros(0, 64, dtype=torch.bfloat16, device=dev()), weight,
                                    torch.zeros(0, dtype=torch.int64, device=dev()))
    assert logp.numel() == 0 and lse.numel() == 0


def test_unsupported_hidden_size_raises():
    with pytest.raises(rlk.RlkError) as e:
        rlk.linear_logp_fwd(torch.zeros(4, 96, dtype=torch.bfloat16, device=dev()),
                            torch.zeros(10, 96, dtype=torch.bfloat16, device=dev()),
                            torch.zeros(4, dtype=torch.int64, device=dev()))
    assert e.value.status == rlk.RLK_ERR_UNSUPPORTED
