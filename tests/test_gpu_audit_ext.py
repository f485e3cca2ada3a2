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


def _slice_scaled(n, seed, scale_of_slice):
    """Audit inputs whose |d| in 4096-element slice s is multiplied by scale_of_slice(s)."""
    new, old, mask = wl.audit_inputs(n, seed)
    d = new.double() - old.double()
    s = torch.arange(n) // 4096
    scale = torch.tensor([scale_of_slice(int(k)) for k in range((n + 4095) // 4096)],
                         dtype=torch.float64)[s]
    new = (old.double() + d * scale).float()
    return new, old, mask


def _fallback_flags(new, old, mask, eps):
    """Which percentiles took the exact fallback: the selection state in the workspace
    after one call (partials 456 x 80 B, padded to 256 B; the sample's histogram of
    4099 u32 and a 16-byte ticket, padded to 256 B; a histogram of 4099 u64, padded to
    256 B; then the state, whose fallback flags are three int32 at byte 48)."""
    d = dev()
    n = len(new)
    ws = torch.zeros(rlk.rlk_dlogp_audit_ext_workspace_bytes(n), dtype=torch.uint8, device=d)
    res = torch.empty(rlk.AUDIT_EXT_RESULT_BYTES, dtype=torch.uint8, device=d)
    rlk.rlk_dlogp_audit_ext(new.to(d), old.to(d), mask.to(d), None, eps, res, ws)
    def up(x):
        return (x + 255) // 256 * 256
    sel_off = up(up(up(456 * 80) + 4099 * 4 + 16) + 4099 * 8)
    return ws[sel_off + 48: sel_off + 60].cpu().view(torch.int32).tolist()


def test_percentiles_where_the_sample_misrepresents_the_batch():
    # 769 slices: the percentile windows come from every sixth slice (0, 6, 12, ...).
    # (a) |d| in the sampled slices is 1e-4 times that of the others: all three ranks lie
    # outside their windows and the exact fallback selects them.  (b) two unsampled
    # slices (0.26 % of the tokens) hold |d| 30 times larger: the p99 rank moves out of
    # its window, the other two stay inside theirs.  (|d| stays below about 2: exp(d)
    # carries the fp32 rounding of d, |d| 2^-24 relative, into mean ratio0.)
    n = 769 * 4096 - 1000
    assert -(-n // 4096) == 769
    new, old, mask = _slice_scaled(n, 31, lambda k: 1e-4 if k % 3 == 0 else 1.0)
    _compare(new, old, mask, None, 0.01)
    assert _fallback_flags(new, old, mask, 0.01) == [1, 1, 1]
    new, old, mask = _slice_scaled(n, 32, lambda k: 30.0 if k in (1, 385) else 1.0)
    _compare(new, old, mask, None, 0.01)
    assert _fallback_flags(new, old, mask, 0.01) == [0, 0, 1]
    # a representative sample: no fallback
    new, old, mask = wl.audit_inputs(n, 34)
    _compare(new, old, mask, None, 0.01)
    assert _fallback_flags(new, old, mask, 0.01) == [0, 0, 0]


def test_windows_open_to_either_side():
    # Few tokens per sampled slice are active: some windows reach the first or the last
    # coarse bin.  Also all active tokens equal, and a NaN among them.
    n = 600 * 4096
    new, old, mask = wl.audit_inputs(n, 33)
    mask[:] = 0
    mask[::4096] = 1
    mask[5::9999] = 1
    _compare(new, old, mask, None, 0.2)
    new2 = old.clone()
    new2[::7] += 0.5
    _compare(new2, old, None, None, 0.2)
    new2[12345] = float("nan")
    _compare(new2, old, None, None, 0.2)
