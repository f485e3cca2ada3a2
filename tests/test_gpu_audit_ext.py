"""Extended dlogp diagnostics ("RL-Kernel integration roadmap for vime",
Consistency Contract: abs_dlogp mean / max / p50 / p90 / p99, ratio0,
clipfrac0, approx_kl0, active count, worst-token location) against the
oracle: counts, worst token and its sequence / position exact; percentiles
equal to the fp32 values the oracle selects (exact order statistics); means
within 1e-6 relative; clip count within the tokens that sit within 1e-6 of the
clip edge (the kernel decides in fp32, the oracle in fp64)."""
import math

import numpy as np
import pytest
import torch

import oracle
import rl_post_linear_gb300 as rlk
import workloads as wl
from helpers import dev

pytestmark = pytest.mark.gpu


def _compare(new, old, mask, offs, eps):
    d = dev()
    r = rlk.dlogp_audit_ext(new.to(d), old.to(d), None if mask is None else mask.to(d),
                            None if offs is None else offs.to(d), eps)
    o = oracle.dlogp_audit_ext(new.numpy(), old.numpy(), None if mask is None else mask.numpy(),
                               None if offs is None else offs.numpy(), eps)
    for k in ("active_count", "argmax_index", "argmax_seq", "argmax_pos"):
        assert r[k] == o[k], k
    if o["active_count"] == 0:
        assert math.isnan(r["p50_abs_dlogp"]) and math.isnan(r["mean_abs_dlogp"])
        return r, o
    for k in ("max_abs_dlogp", "p50_abs_dlogp", "p90_abs_dlogp", "p99_abs_dlogp"):
        assert r[k] == np.float32(o[k]) or (math.isnan(r[k]) and math.isnan(o[k])), k
    for k in ("mean_abs_dlogp", "mean_ratio", "approx_kl"):
        if math.isnan(o[k]):                       # a NaN dlogp among the active tokens
            assert math.isnan(r[k]) and r["error_flags"] & 1, k
        else:
            assert abs(r[k] - o[k]) <= 1e-6 * abs(o[k]) + 1e-15, k
    act = np.ones(len(new), bool) if mask is None else mask.numpy() > 0
    dd = new.double().numpy()[act] - old.double().numpy()[act]
    edge = int(np.sum(np.abs(np.abs(np.exp(dd) - 1) - eps) < 1e-6))
    assert abs(r["clip_count"] - o["clip_count"]) <= edge
    return r, o


@pytest.mark.parametrize("n", [1, 7, 4095, 4097, 100003, 9_400_614])
def test_parity(n):
    new, old, mask = wl.audit_inputs(n, n + 1)
    lens = wl.sweep_lengths(n % 17)[: max(1, min(128, n // 64))]
    offs = np.concatenate([[0], np.cumsum(lens)])
    offs = offs[offs < n]
    offs = torch.from_numpy(np.append(offs, n).astype(np.int64))
    r, o = _compare(new, old, mask, offs, 0.01)
    print("audit ext n=%d: p50 %.3e p90 %.3e p99 %.3e clipfrac %.4f" %
          (n, r["p50_abs_dlogp"], r["p90_abs_dlogp"], r["p99_abs_dlogp"], r["clipfrac"]))


def test_edge_cases():
    z = torch.zeros(50)
    _compare(z, z, torch.zeros(50, dtype=torch.uint8), None, 0.2)
    # ties and a NaN among the active tokens
    new = torch.tensor([0.5, -0.5, 0.25, float("nan"), 0.25, 0.0])
    _compare(new, torch.zeros(6), torch.tensor([1, 1, 1, 0, 1, 1], dtype=torch.uint8), None, 0.2)
    _compare(new, torch.zeros(6), None, torch.tensor([0, 2, 6]), 0.2)
    # many equal values: the selected order statistic is exact
    new = torch.full((20000,), 0.125)
    new[::7] = -0.5
    _compare(new, torch.zeros(20000), None, None, 0.3)
