"""Pins for the fp64 oracle: each check ties it to something other than itself.

Forward: closed forms (W = 0 gives -log V; V = 1 gives 0; V = 2 gives a
log-sigmoid; h = 0 gives a uniform softmax), normalisation (sum over all
targets of exp(logp) = 1), temperature scaling, a logit shift, permutation
equivariance, and high-precision brute force (exact rational dot products,
50-digit exp/log) on vocabularies of at most 16 entries.

Backward: central finite differences of L = sum_t g_t logp_t on tiny shapes,
the softmax-gradient invariant (dW column sums vanish), and closed forms for
h = 0 and W = 0.

Audit and GRPO: hand-built vectors, exact rational means, finite differences
of the clipped objective, and the clip branches.

Full-vocabulary KL against a reference head: identical heads give exactly 0,
swapping the heads swaps the two directions, V = 2 gives the Bernoulli KL of
two log-sigmoids, 60-digit brute force on an 11-entry vocabulary, and central
finite differences of sum g kl + sum gr kl_rev for the backward.

The method is the fused linear selected-token log-prob of "RL-Kernel Roadmap
(2026)" P0.2 and "RL-Kernel integration roadmap for vime" (linear_logp /
lm_head + logp; Consistency Contract for the audit).
"""
import math
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest


def _bf16_grid(rng, shape, scale):
    """random doubles that are exactly representable in bf16."""
    import torch
    x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * np.float32(scale))
    return x.to(torch.bfloat16).double().numpy()


def _fwd(o, h, w, y, mask=None, T=1.0):
    return o.linear_logp_fwd(h, w, np.asarray(y, np.int64), mask, T)


# ----------------------------------------------------------------------------- forward closed forms

def test_zero_weight_gives_minus_log_v(oracle_lib):
    rng = np.random.default_rng(1)
    for vocab in (1, 2, 7, 1000):
        h = _bf16_grid(rng, (5, 16), 1.0)
        w = np.zeros((vocab, 16))
        y = rng.integers(0, vocab, 5)
        logp, lse = _fwd(oracle_lib, h, w, y, T=0.7)
        np.testing.assert_allclose(logp, -math.log(vocab), rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse, math.log(vocab), rtol=0, atol=1e-14)


def test_single_entry_vocab_gives_zero(oracle_lib):
    rng = np.random.default_rng(2)
    h = _bf16_grid(rng, (4, 8), 3.0)
    w = _bf16_grid(rng, (1, 8), 3.0)
    logp, _ = _fwd(oracle_lib, h, w, [0, 0, 0, 0], T=0.3)
    assert np.all(logp == 0.0)


def test_two_entry_vocab_is_log_sigmoid(oracle_lib):
    rng = np.random.default_rng(3)
    h = _bf16_grid(rng, (6, 32), 1.0)
    w = _bf16_grid(rng, (2, 32), 0.3)
    y = np.array([0, 1, 0, 1, 1, 0])
    T = 0.7
    logp, _ = _fwd(oracle_lib, h, w, y, T=T)
    for t in range(6):
        s = [sum(Fraction(a) * Fraction(b) for a, b in zip(h[t], w[v])) for v in range(2)]
        diff = float((s[1 - y[t]] - s[y[t]]) / Fraction(T))
        expect = -math.log1p(math.exp(diff)) if diff < 30 else -diff - math.log1p(math.exp(-diff))
        assert abs(logp[t] - expect) < 1e-13


def test_hand_worked_three_entry_example(oracle_lib):
    # h = (1, 0), W rows (1,0), (0,1), (-1,0): logits (1, 0, -1) at T = 1.
    h = np.array([[1.0, 0.0], [1.0, 0.0], [1.0, 0.0]])
    w = np.array([[1.0, 0.0], [0.0, 1.0], [-1.0, 0.0]])
    logp, lse = _fwd(oracle_lib, h, w, [0, 1, 2], T=1.0)
    z = math.log(math.e + 1.0 + math.exp(-1.0))
    np.testing.assert_allclose(logp, [1.0 - z, -z, -1.0 - z], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, [z, z, z], rtol=0, atol=1e-15)
    # T = 2 halves every logit
    logp2, _ = _fwd(oracle_lib, h, w, [0, 1, 2], T=2.0)
    z2 = math.log(math.exp(0.5) + 1.0 + math.exp(-0.5))
    np.testing.assert_allclose(logp2, [0.5 - z2, -z2, -0.5 - z2], rtol=0, atol=1e-15)


def test_zero_hidden_gives_uniform(oracle_lib):
    rng = np.random.default_rng(4)
    w = _bf16_grid(rng, (37, 16), 1.0)
    logp, _ = _fwd(oracle_lib, np.zeros((3, 16)), w, [0, 5, 36], T=1.3)
    np.testing.assert_allclose(logp, -math.log(37), rtol=0, atol=1e-14)


def test_probabilities_sum_to_one(oracle_lib):
    rng = np.random.default_rng(5)
    vocab, hdim = 300, 24
    h1 = _bf16_grid(rng, (1, hdim), 1.0)
    w = _bf16_grid(rng, (vocab, hdim), 0.5)
    h = np.repeat(h1, vocab, axis=0)
    logp, lse = _fwd(oracle_lib, h, w, np.arange(vocab), T=0.7)
    assert abs(math.fsum(np.exp(logp)) - 1.0) < 1e-13
    assert np.all(lse == lse[0])


def test_temperature_scaling(oracle_lib):
    rng = np.random.default_rng(6)
    h = _bf16_grid(rng, (8, 32), 1.0)
    w = _bf16_grid(rng, (50, 32), 0.2)
    y = rng.integers(0, 50, 8)
    T = 0.7
    a, _ = _fwd(oracle_lib, h, w, y, T=T)
    b, _ = _fwd(oracle_lib, h, w / T, y, T=1.0)
    c, _ = _fwd(oracle_lib, h / T, w, y, T=1.0)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    np.testing.assert_allclose(a, c, rtol=0, atol=1e-12)
    # power-of-two temperature: the scalings are exact
    d, _ = _fwd(oracle_lib, h, w, y, T=4.0)
    e, _ = _fwd(oracle_lib, h, w * 0.25, y, T=1.0)
    np.testing.assert_allclose(d, e, rtol=0, atol=1e-14)
    # T -> infinity flattens the distribution
    f, _ = _fwd(oracle_lib, h, w, y, T=1e12)
    np.testing.assert_allclose(f, -math.log(50), rtol=0, atol=1e-9)


def test_logit_shift_and_permutation(oracle_lib):
    rng = np.random.default_rng(7)
    h = _bf16_grid(rng, (6, 16), 1.0)
    w = _bf16_grid(rng, (40, 16), 0.3)
    y = rng.integers(0, 40, 6)
    a, _ = _fwd(oracle_lib, h, w, y, T=0.9)
    # an extra feature that adds the same constant 3 to every logit
    h2 = np.concatenate([h, np.ones((6, 1))], axis=1)
    w2 = np.concatenate([w, np.full((40, 1), 3.0)], axis=1)
    b, _ = _fwd(oracle_lib, h2, w2, y, T=0.9)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    perm = rng.permutation(40)
    inv = np.argsort(perm)
    c, _ = _fwd(oracle_lib, h, w[perm], inv[y], T=0.9)
    np.testing.assert_allclose(a, c, rtol=0, atol=1e-13)


@pytest.mark.parametrize("vocab", [1, 2, 3, 5, 8, 13, 16])
def test_brute_force_high_precision(oracle_lib, vocab):
    getcontext().prec = 60
    rng = np.random.default_rng(100 + vocab)
    hdim = 12
    h = _bf16_grid(rng, (4, hdim), 2.0)
    w = _bf16_grid(rng, (vocab, hdim), 1.0)
    y = rng.integers(0, vocab, 4)
    T = 0.7
    logp, lse = _fwd(oracle_lib, h, w, y, T=T)
    for t in range(4):
        z = []
        for v in range(vocab):
            s = sum(Fraction(a) * Fraction(b) for a, b in zip(h[t], w[v]))
            q = s / Fraction(T)
            z.append(Decimal(q.numerator) / Decimal(q.denominator))
        total = sum((zz.exp() for zz in z), Decimal(0))
        expect = z[y[t]] - total.ln()          # no max subtraction
        assert abs(float(expect) - logp[t]) < 1e-13 * max(1.0, abs(float(expect)))
        assert abs(float(total.ln()) - lse[t]) < 1e-13 * max(1.0, abs(float(total.ln())))


def test_inactive_and_invalid_rows(oracle_lib):
    rng = np.random.default_rng(8)
    h = _bf16_grid(rng, (5, 8), 1.0)
    h[1, :] = np.nan                                   # NaN padding on an inactive row
    w = _bf16_grid(rng, (10, 8), 1.0)
    y = np.array([3, 999, 4, 10, -1])
    mask = np.array([1, 0, 1, 1, 1], np.uint8)
    logp, lse = oracle_lib.linear_logp_fwd(h, w, y, mask, 1.0)
    assert logp[1] == 0.0 and lse[1] == 0.0
    assert np.isnan(logp[3]) and np.isnan(logp[4])
    assert np.isfinite(logp[0]) and np.isfinite(logp[2])


# ----------------------------------------------------------------------------- backward

def _loss(o, h, w, y, mask, g, T):
    logp, _ = o.linear_logp_fwd(h, w, y, mask, T)
    return float(np.dot(g, np.where(np.isfinite(logp), logp, 0.0)))


@pytest.mark.parametrize("shape", [(1, 3, 2), (3, 5, 4), (4, 8, 6)])
def test_backward_finite_differences(oracle_lib, shape):
    o = oracle_lib
    n, hdim, vocab = shape
    rng = np.random.default_rng(200 + n)
    h = rng.standard_normal((n, hdim))
    w = rng.standard_normal((vocab, hdim)) * 0.7
    y = rng.integers(0, vocab, n)
    mask = np.ones(n, np.uint8)
    if n > 2:
        mask[1] = 0
    g = rng.standard_normal(n)
    T = 0.7
    _, lse = o.linear_logp_fwd(h, w, y, mask, T)
    dh = o.linear_logp_bwd_dh(h, w, y, mask, g, lse, T)
    dw = o.linear_logp_bwd_dw(h, w, y, mask, g, lse, T)
    step = 1e-6
    for arr, grad in ((h, dh), (w, dw)):
        for idx in np.ndindex(arr.shape):
            keep = arr[idx]
            arr[idx] = keep + step
            up = _loss(o, h, w, y, mask, g, T)
            arr[idx] = keep - step
            dn = _loss(o, h, w, y, mask, g, T)
            arr[idx] = keep
            fd = (up - dn) / (2 * step)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, grad[idx])
    if n > 2:
        assert np.all(dh[1] == 0.0)


def test_backward_softmax_invariant(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(9)
    h = _bf16_grid(rng, (12, 16), 1.0)
    w = _bf16_grid(rng, (30, 16), 0.4)
    y = rng.integers(0, 30, 12)
    g = rng.standard_normal(12)
    mask = (rng.random(12) < 0.7).astype(np.uint8)
    _, lse = o.linear_logp_fwd(h, w, y, mask, 0.7)
    dw = o.linear_logp_bwd_dw(h, w, y, mask, g, lse, 0.7)
    # sum_v G[t][v] = 0 for each row, hence sum_v dW_v = 0
    scale = np.abs(dw).sum(axis=0).max()
    assert np.abs(dw.sum(axis=0)).max() < 1e-13 * scale
    # an inactive row's content does not reach dW
    h2 = h.copy()
    h2[mask == 0] = 123.0
    dw2 = o.linear_logp_bwd_dw(h2, w, y, mask, g, lse, 0.7)
    assert np.array_equal(dw, dw2)


def test_backward_closed_forms(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(10)
    vocab, hdim, n, T = 9, 6, 4, 0.7
    w = rng.standard_normal((vocab, hdim))
    y = np.array([0, 3, 3, 8])
    g = rng.standard_normal(n)
    mask = np.ones(n, np.uint8)
    # h = 0: uniform softmax, dh_t = (g_t/T) (W_y - mean_v W_v), dW = 0
    h = np.zeros((n, hdim))
    _, lse = o.linear_logp_fwd(h, w, y, mask, T)
    dh = o.linear_logp_bwd_dh(h, w, y, mask, g, lse, T)
    expect = (g / T)[:, None] * (w[y] - w.mean(axis=0))
    np.testing.assert_allclose(dh, expect, rtol=0, atol=1e-13)
    assert np.all(o.linear_logp_bwd_dw(h, w, y, mask, g, lse, T) == 0.0)
    # W = 0: dW_v = sum_t (g_t/T)(delta - 1/V) h_t, dh = 0
    h = rng.standard_normal((n, hdim))
    w0 = np.zeros((vocab, hdim))
    _, lse = o.linear_logp_fwd(h, w0, y, mask, T)
    dw = o.linear_logp_bwd_dw(h, w0, y, mask, g, lse, T)
    onehot = np.zeros((n, vocab))
    onehot[np.arange(n), y] = 1.0
    expect = ((onehot - 1.0 / vocab) * (g / T)[:, None]).T @ h
    np.testing.assert_allclose(dw, expect, rtol=0, atol=1e-13)
    assert np.all(o.linear_logp_bwd_dh(h, w0, y, mask, g, lse, T) == 0.0)


def test_backward_row_ranges_agree(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(11)
    h = _bf16_grid(rng, (10, 8), 1.0)
    w = _bf16_grid(rng, (20, 8), 0.5)
    y = rng.integers(0, 20, 10)
    g = rng.standard_normal(10)
    _, lse = o.linear_logp_fwd(h, w, y, None, 1.1)
    full = o.linear_logp_bwd_dw(h, w, y, None, g, lse, 1.1)
    part = o.linear_logp_bwd_dw_parallel(h, w, y, None, g, lse, 1.1, 5, 17, threads=3)
    assert np.array_equal(full[5:17], part)
    dh = o.linear_logp_bwd_dh(h, w, y, None, g, lse, 1.1)
    assert np.array_equal(dh, o.linear_logp_bwd_dh_parallel(h, w, y, None, g, lse, 1.1, threads=4))
    lp, ls = o.linear_logp_fwd(h, w, y, None, 1.1)
    lp2, ls2 = o.linear_logp_fwd_parallel(h, w, y, None, 1.1, threads=3)
    assert np.array_equal(lp, lp2) and np.array_equal(ls, ls2)


# ----------------------------------------------------------------------------- audit

def _audit(o, new, old, mask):
    return o.dlogp_audit(np.asarray(new, np.float32), np.asarray(old, np.float32),
                         None if mask is None else np.asarray(mask, np.uint8))


def test_audit_all_masked(oracle_lib):
    r = _audit(oracle_lib, [1, 2, 3], [0, 0, 0], [0, 0, 0])
    assert r["active_count"] == 0 and r["argmax_index"] == -1 and r["max_abs_dlogp"] == 0.0
    assert math.isnan(r["mean_dlogp"]) and math.isnan(r["approx_kl"])
    r = _audit(oracle_lib, [], [], [])
    assert r["active_count"] == 0 and r["argmax_index"] == -1


def test_audit_single_and_ties(oracle_lib):
    r = _audit(oracle_lib, [-1.0, -2.5, -3.0], [-1.0, -2.0, -3.0], [0, 1, 0])
    assert r["active_count"] == 1 and r["argmax_index"] == 1
    assert r["max_abs_dlogp"] == 0.5 and r["mean_dlogp"] == -0.5
    assert abs(r["approx_kl"] - (math.expm1(-0.5) + 0.5)) < 1e-16
    # ties go to the lowest index; masked entries never win
    r = _audit(oracle_lib, [0.0, 0.25, -0.25, 0.25, 9.0], [0.0, 0.0, 0.0, 0.0, 0.0], [1, 1, 1, 1, 0])
    assert r["argmax_index"] == 1 and r["max_abs_dlogp"] == 0.25 and r["active_count"] == 4
    # d = 0 everywhere: zero mean, zero KL
    r = _audit(oracle_lib, [-1.0, -2.0], [-1.0, -2.0], None)
    assert r["mean_dlogp"] == 0.0 and r["approx_kl"] == 0.0 and r["argmax_index"] == 0
    # a NaN ranks above every number
    r = _audit(oracle_lib, [0.0, 5.0, float("nan"), float("nan")], [0.0] * 4, None)
    assert r["argmax_index"] == 2 and math.isnan(r["max_abs_dlogp"])
    # exact |d| that differ below fp32 resolution tie, and the first index wins: the
    # second token's exact |d| = 1.5 + 2^-24 is the larger, but it rounds (to even) to the
    # first token's 1.5
    old = np.array([-3.0, -1.0], np.float32)
    new = np.array([np.float32(-1.5), np.float32(0.5) + np.float32(2.0 ** -24)], np.float32)
    d_exact = [Fraction(float(new[i])) - Fraction(float(old[i])) for i in range(2)]
    d32 = [np.float32(new[i]) - np.float32(old[i]) for i in range(2)]
    assert d_exact[1] > d_exact[0] and d32[0] == d32[1] == np.float32(1.5)
    r = _audit(oracle_lib, new, old, None)
    assert r["argmax_index"] == 0 and r["max_abs_dlogp"] == 1.5


def test_audit_exact_rationals(oracle_lib):
    rng = np.random.default_rng(12)
    n = 5000
    old = (-rng.exponential(1.0, n)).astype(np.float32)
    new = (old + rng.normal(0, 0.01, n)).astype(np.float32)
    mask = (rng.random(n) < 0.8).astype(np.uint8)
    r = _audit(oracle_lib, new, old, mask)
    act = np.nonzero(mask)[0]
    assert r["active_count"] == int(mask.sum())
    d = [Fraction(float(new[t])) - Fraction(float(old[t])) for t in act]
    mean = sum(d, Fraction(0)) / len(d)
    assert abs(r["mean_dlogp"] - float(mean)) <= 1e-15 * float(sum(abs(x) for x in d) / len(d))
    # the worst token is ranked on |d| rounded once to fp32 (the fp32 difference of the logps)
    absd = [float(np.float32(float(abs(x)))) for x in d]
    best = max(absd)
    assert r["max_abs_dlogp"] == best
    assert r["argmax_index"] == int(act[absd.index(best)])
    kl = math.fsum(math.expm1(float(x)) - float(x) for x in d) / len(d)
    assert abs(r["approx_kl"] - kl) < 1e-12 * kl
    # second-order expansion: KL ~ mean d^2 / 2 for small d
    assert abs(r["approx_kl"] - float(np.mean(np.square([float(x) for x in d]))) / 2) < 0.02 * kl


# ----------------------------------------------------------------------------- GRPO objective

def test_grpo_ratio_one_and_clip_branches(oracle_lib):
    o = oracle_lib
    logp = np.array([-1.0, -2.0, -3.0, -0.5, -0.7, -0.9])
    adv = np.array([1.0, -2.0, 0.5, 1.0, 1.0, -1.0])
    mask = np.array([1, 1, 1, 0, 1, 1], np.uint8)
    loss, g = o.grpo_clip_grad(logp, logp.copy(), adv, mask, 0.2)
    na = 5
    np.testing.assert_allclose(g, np.where(mask == 1, -adv / na, 0.0), rtol=0, atol=1e-16)
    assert abs(loss - (-(adv * mask).sum() / na)) < 1e-15
    # r = e^{0.5} > 1.2 with A > 0: clipped branch selected -> zero gradient
    old = logp - np.array([0.5, 0, 0, 0, 0.5, -0.5])
    _, g = o.grpo_clip_grad(logp, old, adv, mask, 0.2)
    assert g[0] == 0.0 and g[4] == 0.0
    # r = e^{-0.5} < 0.8 with A < 0: clipped (constant) selected -> zero gradient
    assert g[5] == 0.0
    # r < 1 - eps with A > 0: unclipped is the minimum -> gradient flows
    old2 = logp + np.array([0.5, 0, 0, 0, 0, 0])
    _, g2 = o.grpo_clip_grad(logp, old2, adv, mask, 0.2)
    assert abs(g2[0] - (-adv[0] * math.exp(-0.5) / na)) < 1e-16


def test_grpo_finite_differences(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(13)
    n = 40
    logp = -rng.exponential(1.0, n)
    old = logp + rng.normal(0, 0.15, n)
    adv = rng.normal(0, 1, n)
    mask = (rng.random(n) < 0.8).astype(np.uint8)
    _, g = o.grpo_clip_grad(logp, old, adv, mask, 0.2)
    step = 1e-7
    for t in range(n):
        r = math.exp(logp[t] - old[t])
        if abs(r - 0.8) < 1e-4 or abs(r - 1.2) < 1e-4:
            continue                                    # kink of the clip
        up = logp.copy()
        up[t] += step
        dn = logp.copy()
        dn[t] -= step
        fd = (o.grpo_clip_grad(up, old, adv, mask, 0.2)[0]
              - o.grpo_clip_grad(dn, old, adv, mask, 0.2)[0]) / (2 * step)
        assert abs(fd - g[t]) < 1e-7, (t, fd, g[t])


def test_golden_hand_example(oracle_lib):
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "hand_example.json")
    ex = json.load(open(path))
    for case in ex["cases"]:
        n = len(case["targets"])
        h = np.repeat(np.array(ex["hidden"]), n, axis=0)
        logp, lse = oracle_lib.linear_logp_fwd(h, np.array(ex["weight"]), case["targets"], None,
                                               case["temperature"])
        np.testing.assert_allclose(logp, case["logp"], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse, case["lse"], rtol=0, atol=1e-15)


def test_grpo_general_reduces_to_symmetric_token_mean(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(14)
    n = 300
    logp = -rng.exponential(1.0, n)
    old = logp + rng.normal(0, 0.2, n)
    adv = rng.normal(0, 1, n)
    mask = (rng.random(n) < 0.7).astype(np.uint8)
    loss, g = o.grpo_clip_grad(logp, old, adv, mask, 0.2)
    g2, res = o.grpo_clip(logp, old, adv, mask, 0.2, 0.2, 1.0 / int(mask.sum()))
    assert np.allclose(g, g2, rtol=1e-15, atol=0) and abs(res["loss"] - loss) < 1e-15
    # counts by direct enumeration
    r = np.exp(logp - old)
    act = mask > 0
    outside = act & ((r < 0.8) | (r > 1.2))
    assert res["active_count"] == act.sum() and res["outside_count"] == outside.sum()
    zero_grad = act & (g2 == 0) & outside
    assert res["clipped_count"] == zero_grad.sum()
    assert abs(res["mean_ratio"] - r[act].mean()) < 1e-14


def test_grpo_general_asymmetric_finite_differences(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(15)
    n = 50
    logp = -rng.exponential(1.0, n)
    old = logp + rng.normal(0, 0.2, n)
    adv = rng.normal(0, 1, n)
    mask = (rng.random(n) < 0.8).astype(np.uint8)
    lo, hi, scale = 0.2, 0.28, 0.013
    g, _ = o.grpo_clip(logp, old, adv, mask, lo, hi, scale)
    step = 1e-7
    for t in range(n):
        r = math.exp(logp[t] - old[t])
        if abs(r - (1 - lo)) < 1e-4 or abs(r - (1 + hi)) < 1e-4:
            continue
        up, dn = logp.copy(), logp.copy()
        up[t] += step
        dn[t] -= step
        fd = (o.grpo_clip(up, old, adv, mask, lo, hi, scale)[1]["loss"]
              - o.grpo_clip(dn, old, adv, mask, lo, hi, scale)[1]["loss"]) / (2 * step)
        assert abs(fd - g[t]) < 1e-8, (t, fd, g[t])
    # an asymmetric range: r = 1.25 is inside [0.8, 1.28] (no clip), outside [0.8, 1.2]
    one = np.array([math.log(1.25)])
    g_in, res_in = o.grpo_clip(one, np.zeros(1), np.ones(1), None, 0.2, 0.28, 1.0)
    g_out, res_out = o.grpo_clip(one, np.zeros(1), np.ones(1), None, 0.2, 0.2, 1.0)
    assert g_in[0] == -1.25 and res_in["outside_count"] == 0
    assert g_out[0] == 0.0 and res_out["clipped_count"] == 1 and abs(res_out["loss"] + 1.2) < 1e-15


# ----------------------------------------------------------------------------- logp from logits

def test_logits_closed_forms(oracle_lib):
    o = oracle_lib
    # equal logits -> -log V; two entries -> log-sigmoid of the gap; the hand example
    z = np.zeros((3, 37))
    logp, lse = o.logp_from_logits(z + 5.0, [0, 7, 36], None, 0.7)
    np.testing.assert_allclose(logp, -math.log(37), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, 5.0 / 0.7 + math.log(37), rtol=0, atol=1e-13)
    z2 = np.array([[0.3, -1.1], [2.0, 2.5]])
    logp, _ = o.logp_from_logits(z2, [1, 0], None, 0.5)
    for i, (a, b) in enumerate(z2):
        mine, other = (b, a) if i == 0 else (a, b)
        assert abs(logp[i] + math.log1p(math.exp((other - mine) / 0.5))) < 1e-14
    ex = np.array([[1.0, 0.0, -1.0]])
    logp, lse = o.logp_from_logits(ex, [0], None, 1.0)
    assert abs(lse[0] - math.log(math.e + 1 + math.exp(-1))) < 1e-15


def test_logits_brute_force_and_normalisation(oracle_lib):
    getcontext().prec = 60
    o = oracle_lib
    rng = np.random.default_rng(20)
    z = rng.standard_normal((4, 13)) * 3
    y = rng.integers(0, 13, 4)
    logp, _ = o.logp_from_logits(z, y, None, 0.7)
    for t in range(4):
        d = [Decimal(float(v)) / Decimal(0.7) for v in z[t]]
        tot = sum((x.exp() for x in d), Decimal(0))
        assert abs(float(d[y[t]] - tot.ln()) - logp[t]) < 1e-13
    allv, _ = o.logp_from_logits(np.repeat(z[:1], 13, axis=0), np.arange(13), None, 1.3)
    assert abs(math.fsum(np.exp(allv)) - 1.0) < 1e-13


def test_logits_indexed_rows_and_mask(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(21)
    z = rng.standard_normal((10, 50))
    y = rng.integers(0, 50, 10)
    mask = np.array([1, 1, 0, 1, 1, 1, 1, 0, 1, 1], np.uint8)
    dense, dlse = o.logp_from_logits(z, y, mask, 0.9)
    rows = np.array([9, 2, 4, 4, 0])
    idx, ilse = o.logp_from_logits(z, y, mask, 0.9, rows=rows)
    assert np.array_equal(idx, dense[rows]) and np.array_equal(ilse, dlse[rows])
    assert dense[2] == 0.0 and dense[7] == 0.0
    y2 = y.copy()
    y2[3] = 50
    bad, _ = o.logp_from_logits(z, y2, mask, 0.9)
    assert math.isnan(bad[3])


# ----------------------------------------------------------------------------- entropy

def test_entropy_closed_forms(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(30)
    h = _bf16_grid(rng, (4, 16), 1.0)
    # W = 0: uniform softmax, entropy = log V; V = 1: entropy 0
    _, _, ent = o.linear_logp_entropy_fwd(h, np.zeros((50, 16)), [0, 1, 2, 3], None, 0.7)
    np.testing.assert_allclose(ent, math.log(50), rtol=0, atol=1e-13)
    _, _, ent1 = o.linear_logp_entropy_fwd(h, _bf16_grid(rng, (1, 16), 1.0), [0] * 4, None, 0.7)
    assert np.all(np.abs(ent1) < 1e-15)
    # V = 2: binary entropy of sigmoid(gap)
    w2 = _bf16_grid(rng, (2, 16), 0.4)
    lp, _, ent2 = o.linear_logp_entropy_fwd(h, w2, [0] * 4, None, 1.3)
    p0 = np.exp(lp)
    np.testing.assert_allclose(ent2, -(p0 * np.log(p0) + (1 - p0) * np.log1p(-p0)), rtol=1e-12)
    # logp and lse agree with the logp-only forward
    w = _bf16_grid(rng, (40, 16), 0.5)
    y = rng.integers(0, 40, 4)
    a, b, _ = o.linear_logp_entropy_fwd(h, w, y, None, 0.9)
    c, d = o.linear_logp_fwd(h, w, y, None, 0.9)
    assert np.array_equal(a, c) and np.array_equal(b, d)


def test_entropy_brute_force(oracle_lib):
    getcontext().prec = 60
    o = oracle_lib
    rng = np.random.default_rng(31)
    h = _bf16_grid(rng, (3, 10), 2.0)
    w = _bf16_grid(rng, (9, 10), 1.0)
    _, _, ent = o.linear_logp_entropy_fwd(h, w, [0, 1, 2], None, 0.7)
    for t in range(3):
        z = []
        for v in range(9):
            q = sum(Fraction(a) * Fraction(b) for a, b in zip(h[t], w[v])) / Fraction(0.7)
            z.append(Decimal(q.numerator) / Decimal(q.denominator))
        tot = sum((x.exp() for x in z), Decimal(0))
        expect = -sum(((x.exp() / tot) * (x - tot.ln()) for x in z), Decimal(0))
        assert abs(float(expect) - ent[t]) < 1e-13


@pytest.mark.parametrize("shape", [(2, 3, 4), (3, 6, 5)])
def test_entropy_backward_finite_differences(oracle_lib, shape):
    o = oracle_lib
    n, hdim, vocab = shape
    rng = np.random.default_rng(40 + n)
    h = rng.standard_normal((n, hdim))
    w = rng.standard_normal((vocab, hdim)) * 0.7
    y = rng.integers(0, vocab, n)
    mask = np.ones(n, np.uint8)
    mask[-1] = 0 if n > 2 else 1
    g, gh = rng.standard_normal(n), rng.standard_normal(n)
    T = 0.8

    def loss():
        lp, _, ent = o.linear_logp_entropy_fwd(h, w, y, mask, T)
        return float(np.dot(g, lp) + np.dot(gh, ent))

    _, lse, ent = o.linear_logp_entropy_fwd(h, w, y, mask, T)
    dh = o.linear_logp_entropy_bwd_dh(h, w, y, mask, g, gh, lse, ent, T)
    dw = o.linear_logp_entropy_bwd_dw(h, w, y, mask, g, gh, lse, ent, T)
    step = 1e-6
    for arr, grad in ((h, dh), (w, dw)):
        for idx in np.ndindex(arr.shape):
            keep = arr[idx]
            arr[idx] = keep + step
            up = loss()
            arr[idx] = keep - step
            dn = loss()
            arr[idx] = keep
            fd = (up - dn) / (2 * step)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, grad[idx])
    # gH = 0 reduces to the logp-only backward
    z = np.zeros(n)
    assert np.allclose(o.linear_logp_entropy_bwd_dw(h, w, y, mask, g, z, lse, ent, T),
                       o.linear_logp_bwd_dw(h, w, y, mask, g, lse, T), rtol=1e-14, atol=1e-15)


# ----------------------------------------------------------------------------- extended audit

def test_audit_ext_hand_built(oracle_lib):
    o = oracle_lib
    # |d| = 1..100 (a permutation), all active: nearest-rank p50 = 50, p90 = 90, p99 = 99
    perm = np.random.default_rng(0).permutation(100)
    d = (perm + 1).astype(np.float32) * np.float32(0.001)
    sign = np.where(np.arange(100) % 2 == 0, 1, -1).astype(np.float32)
    r = o.dlogp_audit_ext(d * sign, np.zeros(100, np.float32), None, None, 0.05)
    srt = np.sort(d.astype(np.float64))
    assert r["p50_abs_dlogp"] == srt[49] and r["p90_abs_dlogp"] == srt[89]
    assert r["p99_abs_dlogp"] == srt[98] and r["max_abs_dlogp"] == srt[99]
    assert abs(r["mean_abs_dlogp"] - float(np.mean(d.astype(np.float64)))) < 1e-15
    # clip: |exp(d) - 1| > 0.05 <=> d > log(1.05) = 0.04879 or d < log(0.95) = -0.05129
    dd = (d * sign).astype(np.float64)
    assert r["clip_count"] == int(np.sum(np.abs(np.exp(dd) - 1) > 0.05))
    assert abs(r["clipfrac"] - r["clip_count"] / 100) < 1e-15
    assert abs(r["mean_ratio"] - float(np.mean(np.exp(dd)))) < 1e-15
    # worst token's sequence and position
    offs = np.array([0, 30, 31, 100], np.int64)
    r = o.dlogp_audit_ext(d * sign, np.zeros(100, np.float32), None, offs, 0.05)
    w = int(np.argmax(d))
    s = int(np.searchsorted(offs, w, side="right") - 1)
    assert r["argmax_index"] == w and r["argmax_seq"] == s and r["argmax_pos"] == w - offs[s]


def test_audit_ext_ratio_and_clip_closed_forms(oracle_lib):
    """ratio0 = exp(logp_new - logp_old) and clipfrac0 counts |ratio0 - 1| > eps ("RL-Kernel
    integration roadmap for vime", Consistency Contract, minimum diagnostics).  With d = ln 2,
    ln 4, ln 1/2 and 0 the ratios are 2, 4, 1/2 and 1: mean 15/8.  A reversed difference gives
    15/16, a ratio of exp|d| gives 9/4; eps = 0.75 clips 2 tokens, while a test on |d| clips 1."""
    o = oracle_lib
    lnv = np.array([math.log(2.0), math.log(4.0), math.log(0.5), 0.0], np.float32)
    for new, old in ((lnv, np.zeros(4, np.float32)), (np.zeros(4, np.float32), -lnv)):
        r = o.dlogp_audit_ext(new, old, None, None, 0.75)
        assert abs(r["mean_ratio"] - 1.875) < 1e-6
        assert r["clip_count"] == 2 and r["clipfrac"] == 0.5
        r = o.dlogp_audit_ext(new, old, None, None, 0.4)
        assert r["clip_count"] == 3
    # a masked-out token contributes to neither
    r = o.dlogp_audit_ext(lnv, np.zeros(4, np.float32), np.array([1, 0, 1, 1], np.uint8), None,
                          0.75)
    assert abs(r["mean_ratio"] - 3.5 / 3) < 1e-6 and r["clip_count"] == 1


def test_audit_ext_small_counts_and_masked(oracle_lib):
    o = oracle_lib
    # one active token: every percentile is that token
    r = o.dlogp_audit_ext(np.array([0.5, 0.25, 7.0], np.float32), np.zeros(3, np.float32),
                          np.array([0, 1, 0], np.uint8))
    assert r["p50_abs_dlogp"] == r["p99_abs_dlogp"] == r["max_abs_dlogp"] == 0.25
    # two tokens: p50 is the smaller (rank 1), p90 / p99 the larger (rank 2)
    r = o.dlogp_audit_ext(np.array([-0.3, 0.1], np.float32), np.zeros(2, np.float32), None)
    assert r["p50_abs_dlogp"] == float(np.float32(0.1)) and r["p90_abs_dlogp"] == float(np.float32(0.3))
    # none active
    r = o.dlogp_audit_ext(np.zeros(4, np.float32), np.zeros(4, np.float32), np.zeros(4, np.uint8))
    assert r["active_count"] == 0 and math.isnan(r["p50_abs_dlogp"]) and r["argmax_seq"] == -1
    # a NaN ranks above every number, so it is the p99 / max of a short list
    r = o.dlogp_audit_ext(np.array([0.1, float("nan"), 0.2], np.float32), np.zeros(3, np.float32),
                          None)
    assert math.isnan(r["p99_abs_dlogp"]) and r["p50_abs_dlogp"] == float(np.float32(0.2))


# ----------------------------------------------------------------------------- full-vocabulary KL

def test_kl_identical_heads_and_swap(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(50)
    h, hr = _bf16_grid(rng, (4, 12), 1.0), _bf16_grid(rng, (4, 6), 1.0)
    w, wr = _bf16_grid(rng, (30, 12), 0.5), _bf16_grid(rng, (30, 6), 0.5)
    # the same head on both sides: both divergences vanish exactly, the lse is the logp-only one
    kl, kr, lse, lse_r = o.linear_kl_fwd(h, w, h, w, None, 0.8, 0.8)
    assert np.all(kl == 0) and np.all(kr == 0) and np.array_equal(lse, lse_r)
    _, lse0 = o.linear_logp_fwd(h, w, np.zeros(4, np.int64), None, 0.8)
    assert np.array_equal(lse, lse0)
    # swapping the heads swaps the two directions; both are non-negative
    a = o.linear_kl_fwd(h, w, hr, wr, None, 0.8, 1.4)
    b = o.linear_kl_fwd(hr, wr, h, w, None, 1.4, 0.8)
    assert np.array_equal(a[0], b[1]) and np.array_equal(a[1], b[0])
    assert np.all(a[0] > 0) and np.all(a[1] > 0)
    # masked rows are all zero
    m = np.array([1, 0, 1, 0], np.uint8)
    c = o.linear_kl_fwd(h, w, hr, wr, m, 0.8, 1.4)
    assert all(np.all(x[m == 0] == 0) for x in c)
    assert all(np.array_equal(x[m == 1], y[m == 1]) for x, y in zip(c, a))


def test_kl_two_entry_vocab_is_bernoulli_kl(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(51)
    h, hr = _bf16_grid(rng, (5, 8), 1.0), _bf16_grid(rng, (5, 8), 1.0)
    w, wr = _bf16_grid(rng, (2, 8), 0.6), _bf16_grid(rng, (2, 8), 0.6)
    T, Tr = 0.9, 1.2
    kl, kr, _, _ = o.linear_kl_fwd(h, w, hr, wr, None, T, Tr)
    for t in range(5):
        a = (h[t] @ (w[1] - w[0])) / T                  # logit gap of the policy
        b = (hr[t] @ (wr[1] - wr[0])) / Tr              # and of the reference
        p1, q1 = 1 / (1 + math.exp(-a)), 1 / (1 + math.exp(-b))
        ls = lambda x: -math.log1p(math.exp(-x))        # log sigmoid
        lp1, lp0, lq1, lq0 = ls(a), ls(-a), ls(b), ls(-b)
        f = p1 * (lp1 - lq1) + (1 - p1) * (lp0 - lq0)
        r = q1 * (lq1 - lp1) + (1 - q1) * (lq0 - lp0)
        assert abs(kl[t] - f) <= 1e-13 and abs(kr[t] - r) <= 1e-13


def test_kl_brute_force_high_precision(oracle_lib):
    getcontext().prec = 60
    o = oracle_lib
    rng = np.random.default_rng(52)
    h, hr = _bf16_grid(rng, (3, 10), 2.0), _bf16_grid(rng, (3, 7), 2.0)
    w, wr = _bf16_grid(rng, (11, 10), 0.7), _bf16_grid(rng, (11, 7), 0.7)
    T, Tr = 0.7, 1.1
    kl, kr, lse, lse_r = o.linear_kl_fwd(h, w, hr, wr, None, T, Tr)

    def logits(x, m, temp):
        out = []
        for v in range(m.shape[0]):
            q = sum(Fraction(a) * Fraction(b) for a, b in zip(x, m[v])) / Fraction(temp)
            out.append(Decimal(q.numerator) / Decimal(q.denominator))
        return out

    for t in range(3):
        z, r = logits(h[t], w, T), logits(hr[t], wr, Tr)
        zs = sum((x.exp() for x in z), Decimal(0))
        rs = sum((x.exp() for x in r), Decimal(0))
        lp = [x - zs.ln() for x in z]
        lq = [x - rs.ln() for x in r]
        f = sum((a.exp() * (a - b) for a, b in zip(lp, lq)), Decimal(0))
        b_ = sum((b.exp() * (b - a) for a, b in zip(lp, lq)), Decimal(0))
        assert abs(float(f) - kl[t]) < 1e-13 and abs(float(b_) - kr[t]) < 1e-13
        assert abs(float(zs.ln()) - lse[t]) < 1e-13 and abs(float(rs.ln()) - lse_r[t]) < 1e-13


@pytest.mark.parametrize("shape", [(2, 3, 4, 2), (3, 5, 6, 4)])
def test_kl_backward_finite_differences(oracle_lib, shape):
    o = oracle_lib
    n, hdim, vocab, hrdim = shape
    rng = np.random.default_rng(60 + n)
    h, hr = rng.standard_normal((n, hdim)), rng.standard_normal((n, hrdim))
    w, wr = rng.standard_normal((vocab, hdim)) * 0.7, rng.standard_normal((vocab, hrdim))
    mask = np.ones(n, np.uint8)
    mask[0] = 0 if n > 2 else 1
    g, gr = rng.standard_normal(n), rng.standard_normal(n)
    T, Tr = 0.8, 1.3

    def loss():
        kl, kr, _, _ = o.linear_kl_fwd(h, w, hr, wr, mask, T, Tr)
        return float(np.dot(g, kl) + np.dot(gr, kr))

    kl, _, lse, lse_r = o.linear_kl_fwd(h, w, hr, wr, mask, T, Tr)
    dh = o.linear_kl_bwd_dh(h, w, hr, wr, mask, g, gr, lse, lse_r, kl, T, Tr)
    dw = o.linear_kl_bwd_dw(h, w, hr, wr, mask, g, gr, lse, lse_r, kl, T, Tr)
    step = 1e-6
    for arr, grad in ((h, dh), (w, dw)):
        for idx in np.ndindex(arr.shape):
            keep = arr[idx]
            arr[idx] = keep + step
            up = loss()
            arr[idx] = keep - step
            dn = loss()
            arr[idx] = keep
            fd = (up - dn) / (2 * step)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, grad[idx])
    # the reference head gets no gradient, and every row of G sums to zero, so the dW columns do
    assert np.abs(dw.sum(axis=0)).max() <= 1e-12 * max(1.0, np.abs(dw).max())
