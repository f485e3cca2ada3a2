"""Edge shapes and numerically hard inputs against the fp64 oracle.

* Temperatures far from 1 (T = 0.05 sharpens the softmax to |logp| ~ 100;
  T = 50 flattens it to about -log V) and logits of magnitude ~ 100 at T = 1,
  where an unshifted exp would overflow fp32: the online max / sum-exp must
  keep every term in range ("RL-Kernel integration roadmap for vime",
  linear_logp: temperature applied before the softmax; log-softmax contract).
* A 262144-entry vocabulary (eight backward chunks, 256 forward chunks) and a
  16384-wide hidden size (256 K-steps per tile), forward and backward.
* A confident policy whose sampled token carries most of the mass, and (the
  sharp and large-logit cases, with uniformly drawn targets) rows dominated by
  an entry that is not the target: both dominant entries must keep their
  small gradient parts g (1 - p) / T out of a bf16 difference.
"""
import numpy as np
import pytest
import torch

import oracle
import rl_post_linear_gb300 as rlk
import workloads as wl
from helpers import GRAD_REL_L2, LOGP_ATOL, dev, f64, rel_l2

pytestmark = pytest.mark.gpu


def _inputs(n, h, v, seed, std, active=0.9):
    hidden = wl.normal_bf16((n, h), seed, wl.S_HIDDEN)
    weight = wl.normal_bf16((v, h), seed, wl.S_WEIGHT, std=std)
    targets = wl.uniform_targets(n, v, seed)
    rng = np.random.default_rng(seed)
    mask = torch.from_numpy((rng.random(n) < active).astype(np.uint8))
    grad = rng.standard_normal(n) / n
    grad[mask.numpy() == 0] = 0.0
    return hidden, weight, targets, mask, grad


def _gpu(hidden, weight, targets, mask, grad, T):
    d = dev()
    h, w, y, m = hidden.to(d), weight.to(d), targets.to(d), mask.to(d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    logp, lse = rlk.linear_logp_fwd(h, w, y, m, T, err)
    out = [logp.cpu(), lse.cpu()]
    if grad is not None:
        g = torch.tensor(grad, dtype=torch.float32, device=d)
        dh, dw = rlk.linear_logp_bwd(h, w, y, m, g, lse, T, err)
        out += [dh.cpu(), dw.cpu()]
    torch.cuda.synchronize()
    return out, int(err.item())


def _check_fwd(hidden, weight, targets, mask, T, logp, lse):
    lp_o, lse_o = oracle.linear_logp_fwd_parallel(f64(hidden), f64(weight), targets.numpy(),
                                                  mask.numpy(), T)
    act = mask.numpy() > 0
    dl = np.abs(logp.double().numpy() - lp_o)[act].max()
    dz = np.abs(lse.double().numpy() - lse_o)[act].max()
    return dl, dz, lp_o, lse_o


@pytest.mark.parametrize("T,std,label", [(0.05, 0.1, "sharp"), (50.0, 0.1, "flat"),
                                         (1.0, 2.0, "large logits")])
def test_extreme_temperature_and_magnitude(T, std, label):
    n, h, v = 200, 256, 3000
    hidden, weight, targets, mask, grad = _inputs(n, h, v, 17, std)
    (logp, lse, dh, dw), err = _gpu(hidden, weight, targets, mask, grad, T)
    assert err == 0
    assert torch.isfinite(logp).all() and torch.isfinite(lse).all()
    dl, dz, lp_o, lse_o = _check_fwd(hidden, weight, targets, mask, T, logp, lse)
    act = mask.numpy() > 0
    print("%s (T=%g, W std %g): logp in [%.1f, %.2f], max |dlogp| %.3e, max |dlse| %.3e"
          % (label, T, std, lp_o[act].min(), lp_o[act].max(), dl, dz))
    assert dl <= LOGP_ATOL and dz <= LOGP_ATOL
    h64, w64 = f64(hidden), f64(weight)
    dh_o = oracle.linear_logp_bwd_dh_parallel(h64, w64, targets.numpy(), mask.numpy(), grad,
                                              lse_o, T)
    dw_o = oracle.linear_logp_bwd_dw_parallel(h64, w64, targets.numpy(), mask.numpy(), grad,
                                              lse_o, T, 0, v)
    e_dh, e_dw = rel_l2(dh, dh_o), rel_l2(dw, dw_o)
    print("%s: rel-L2 dh %.3e dw %.3e" % (label, e_dh, e_dw))
    assert e_dh <= GRAD_REL_L2 and e_dw <= GRAD_REL_L2


def test_flat_softmax_reaches_minus_log_v():
    # at T = 1e4 every logit is within ~1e-3 of the others: logp -> -log V
    n, h, v = 64, 128, 5000
    hidden, weight, targets, mask, _ = _inputs(n, h, v, 18, 0.02, active=1.0)
    (logp, _), err = _gpu(hidden, weight, targets, mask, None, 1e4)
    assert err == 0
    assert float((logp.double() + np.log(v)).abs().max()) < 1e-4


def test_large_vocabulary_forward_and_backward():
    n, h, v = 300, 256, 262144
    hidden, weight, targets, mask, grad = _inputs(n, h, v, 19, 0.05)
    (logp, lse, dh, dw), err = _gpu(hidden, weight, targets, mask, grad, 0.8)
    assert err == 0
    dl, dz, _, lse_o = _check_fwd(hidden, weight, targets, mask, 0.8, logp, lse)
    h64, w64 = f64(hidden), f64(weight)
    dh_o = oracle.linear_logp_bwd_dh_parallel(h64, w64, targets.numpy(), mask.numpy(), grad,
                                              lse_o, 0.8)
    dw_o = oracle.linear_logp_bwd_dw_parallel(h64, w64, targets.numpy(), mask.numpy(), grad,
                                              lse_o, 0.8, 0, v)
    e_dh, e_dw = rel_l2(dh, dh_o), rel_l2(dw, dw_o)
    print("V=262144: max |dlogp| %.3e, rel-L2 dh %.3e dw %.3e" % (dl, e_dh, e_dw))
    assert dl <= LOGP_ATOL and dz <= LOGP_ATOL
    assert e_dh <= GRAD_REL_L2 and e_dw <= GRAD_REL_L2


def test_wide_hidden_forward_and_backward():
    n, h, v = 150, 16384, 2000
    hidden, weight, targets, mask, grad = _inputs(n, h, v, 20, 0.01)
    (logp, lse, dh, dw), err = _gpu(hidden, weight, targets, mask, grad, 1.0)
    assert err == 0
    dl, dz, _, lse_o = _check_fwd(hidden, weight, targets, mask, 1.0, logp, lse)
    h64, w64 = f64(hidden), f64(weight)
    dh_o = oracle.linear_logp_bwd_dh_parallel(h64, w64, targets.numpy(), mask.numpy(), grad,
                                              lse_o, 1.0)
    dw_o = oracle.linear_logp_bwd_dw_parallel(h64, w64, targets.numpy(), mask.numpy(), grad,
                                              lse_o, 1.0, 0, v)
    e_dh, e_dw = rel_l2(dh, dh_o), rel_l2(dw, dw_o)
    print("H=16384: max |dlogp| %.3e, rel-L2 dh %.3e dw %.3e" % (dl, e_dh, e_dw))
    assert dl <= LOGP_ATOL and dz <= LOGP_ATOL
    assert e_dh <= GRAD_REL_L2 and e_dw <= GRAD_REL_L2


def test_confident_policy_where_the_target_dominates():
    # A policy late in RL training puts most of the mass on the token it sampled: here each
    # target is its row's argmax and p_y spans ~0.5 to ~1.  The target's gradient entry
    # g (1 - p_y) / T is then much smaller than g / T and g p_y / T, so it must not come out
    # as the difference of those two in low precision.
    n, h, v, T = 256, 256, 3000, 1.0
    hidden, weight, _, mask, grad = _inputs(n, h, v, 23, 1.0)
    logits = hidden.float() @ weight.float().T
    targets = logits.argmax(dim=1)
    (logp, lse, dh, dw), err = _gpu(hidden, weight, targets, mask, grad, T)
    assert err == 0
    dl, dz, lp_o, lse_o = _check_fwd(hidden, weight, targets, mask, T, logp, lse)
    act = mask.numpy() > 0
    p_y = np.exp(lp_o[act])
    h64, w64 = f64(hidden), f64(weight)
    dh_o = oracle.linear_logp_bwd_dh_parallel(h64, w64, targets.numpy(), mask.numpy(), grad,
                                              lse_o, T)
    dw_o = oracle.linear_logp_bwd_dw_parallel(h64, w64, targets.numpy(), mask.numpy(), grad,
                                              lse_o, T, 0, v)
    e_dh, e_dw = rel_l2(dh, dh_o), rel_l2(dw, dw_o)
    print("confident policy: p_y quartiles %s, max |dlogp| %.3e, rel-L2 dh %.3e dw %.3e"
          % (np.round(np.quantile(p_y, [0.0, 0.25, 0.5, 0.75, 1.0]), 4), dl, e_dh, e_dw))
    assert np.median(p_y) > 0.9
    assert dl <= LOGP_ATOL and dz <= LOGP_ATOL
    assert e_dh <= GRAD_REL_L2 and e_dw <= GRAD_REL_L2
