"""GPU clipped-ratio loss fragment vs the oracle ("RL-Kernel integration roadmap
for vime", RL Loss Operators).

Per token: grad within 1e-6 relative of the oracle's; aggregates: loss and mean
ratio within 1e-6 relative, counts exact.  The clip branch is a decision taken
in floating point: the kernel takes it in fp32, the oracle in fp64, so a token
whose fp64 ratio lies within 1e-6 of a clip edge may land on either side.  For
those tokens either branch is accepted (the gradient is checked to be one of
the two valid values) and the counts may differ by at most their number.
"""
import numpy as np
import pytest
import torch

import oracle
import rl_post_linear_gb300 as rlk
import workloads as wl
from helpers import dev

pytestmark = pytest.mark.gpu


def _inputs(n, seed, noise=0.15):
    g = np.random.default_rng(seed)
    old = (-g.exponential(1.0, n)).astype(np.float32)
    new = (old + g.normal(0, noise, n)).astype(np.float32)
    adv = g.normal(0, 1, n).astype(np.float32)
    mask = (g.random(n) < 0.85).astype(np.uint8)
    return new, old, adv, mask


def _check(new, old, adv, mask, lo, hi, scale):
    d = dev()
    t = [torch.from_numpy(x).to(d) for x in (new, old, adv, mask)]
    grad, res = rlk.grpo_clip_loss(t[0], t[1], t[2], t[3], lo, hi, scale)
    g_o, r_o = oracle.grpo_clip(new.astype(np.float64), old.astype(np.float64),
                                adv.astype(np.float64), mask, lo, hi, scale)
    g = grad.cpu().double().numpy()
    r = np.exp(new.astype(np.float64) - old.astype(np.float64))
    edge = (np.abs(r - (1 - lo)) < 1e-6) | (np.abs(r - (1 + hi)) < 1e-6)
    ok = ~edge
    assert np.all(np.abs(g - g_o)[ok] <= 1e-6 * np.abs(g_o)[ok] + 1e-30)
    alt = -scale * adv.astype(np.float64) * r
    for i in np.nonzero(edge & (mask > 0))[0]:
        assert g[i] == 0.0 or abs(g[i] - alt[i]) <= 1e-6 * abs(alt[i])
    assert np.all(g[mask == 0] == 0.0)
    n_edge = int((edge & (mask > 0)).sum())
    assert res["active_count"] == r_o["active_count"] == int(mask.sum())
    assert abs(res["clipped_count"] - r_o["clipped_count"]) <= n_edge
    assert abs(res["outside_count"] - r_o["outside_count"]) <= n_edge
    tol = 1e-6 * scale * float(np.sum(np.abs(adv.astype(np.float64) * r)[mask > 0])) + 1e-12
    assert abs(res["loss"] - r_o["loss"]) <= tol + n_edge * scale * 2.5
    if r_o["active_count"] == 0:
        assert np.isnan(res["mean_ratio"]) and np.isnan(r_o["mean_ratio"]) and res["loss"] == 0.0
    else:
        assert abs(res["mean_ratio"] - r_o["mean_ratio"]) <= 1e-6 * r_o["mean_ratio"]
    return grad, res


@pytest.mark.parametrize("n", [1, 100, 8191, 8192, 8193, 100003])
def test_parity_symmetric_token_mean(n):
    new, old, adv, mask = _inputs(n, n)
    na = max(int(mask.sum()), 1)
    _check(new, old, adv, mask, 0.2, 0.2, 1.0 / na)


def test_parity_asymmetric_and_unaligned():
    new, old, adv, mask = _inputs(50_001, 7, noise=0.3)
    _check(new, old, adv, mask, 0.2, 0.28, 1e-3)
    _check(new[1:], old[1:], adv[1:], mask[1:], 0.1, 0.3, 0.5)


def test_grpo_workload_and_batch_invariance():
    # the benchmark's recipe: old = logp + N(0, 0.01^2), advantages per sequence
    n, lens = 8192, wl.packed_lengths(8192, 8, 512, 2048, 0)
    noise, adv = wl.grpo_bwd_extras(n, lens, 0)
    logp = (-np.random.default_rng(1).exponential(1.0, n)).astype(np.float32)
    old = (logp + noise).astype(np.float32)
    mask = np.ones(n, np.uint8)
    grad, res = _check(logp, old, adv.astype(np.float32), mask, wl.GRPO_EPS, wl.GRPO_EPS, 1.0 / n)
    # with the caller's scale fixed, a token's gradient does not depend on its batch
    d = dev()
    sub = slice(1000, 3333)
    g2, _ = rlk.grpo_clip_loss(*(torch.from_numpy(x[sub]).to(d) for x in
                                 (logp, old, adv.astype(np.float32), mask)),
                               wl.GRPO_EPS, wl.GRPO_EPS, 1.0 / n)
    assert torch.equal(g2.cpu().view(torch.int32), grad[sub].cpu().view(torch.int32))


def test_argument_errors():
    z = torch.zeros(4, device=dev())
    with pytest.raises(rlk.RlkError):
        rlk.grpo_clip_loss(z, z, z, None, 0.2, 0.2, 0.0)
    with pytest.raises(rlk.RlkError):
        rlk.grpo_clip_loss(z, z, z, None, 1.5, 0.2, 1.0)
