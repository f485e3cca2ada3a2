"""GPU dlogp audit vs the oracle ("RL-Kernel integration roadmap for vime",
Consistency Contract): exact counts and worst-token index, max|d| equal to the
fp32 rounding of the oracle's exact difference, mean and approx-KL within
1e-6 relative (mean: relative to mean |d|), bitwise reproducibility.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import rl_post_linear_gb300 as rlk
import workloads as wl
from helpers import dev

pytestmark = pytest.mark.gpu


def _both(new, old, mask):
    d = dev()
    r = rlk.dlogp_audit(new.to(d), old.to(d), None if mask is None else mask.to(d))
    o = oracle.dlogp_audit(new.numpy(), old.numpy(), None if mask is None else mask.numpy())
    return r, o


def _check(r, o, new, old, mask):
    assert r["active_count"] == o["active_count"]
    assert r["argmax_index"] == o["argmax_index"]
    assert r["max_abs_dlogp"] == np.float32(o["max_abs_dlogp"])
    if o["active_count"] == 0:
        assert math.isnan(r["mean_dlogp"]) and math.isnan(r["approx_kl"])
        return
    act = np.ones(len(new), bool) if mask is None else mask.numpy() > 0
    mean_abs = np.mean(np.abs(new.double().numpy() - old.double().numpy())[act])
    assert abs(r["mean_dlogp"] - o["mean_dlogp"]) <= 1e-6 * mean_abs + 1e-12
    assert abs(r["approx_kl"] - o["approx_kl"]) <= 1e-6 * abs(o["approx_kl"]) + 1e-15


@pytest.mark.parametrize("n", [1, 5, 4095, 4096, 4097, 8191, 8192, 8193, 100003])
def test_parity_random(n):
    new, old, mask = wl.audit_inputs(n, n)
    r, o = _both(new, old, mask)
    _check(r, o, new, old, mask)
    r2, _ = _both(new, old, None)
    o2 = oracle.dlogp_audit(new.numpy(), old.numpy(), None)
    _check(r2, o2, new, old, None)


def test_unaligned_inputs_take_the_scalar_path():
    new, old, mask = wl.audit_inputs(50001, 3)
    d = dev()
    nb, ob, mb = new.to(d), old.to(d), mask.to(d)
    r = rlk.dlogp_audit(nb[1:], ob[1:], mb[1:])
    o = oracle.dlogp_audit(new.numpy()[1:], old.numpy()[1:], mask.numpy()[1:])
    _check(r, o, new[1:], old[1:], mask[1:])


def test_degenerate_cases():
    z = torch.zeros(10)
    r, o = _both(z, z, torch.zeros(10, dtype=torch.uint8))
    assert r["active_count"] == 0 and r["argmax_index"] == -1 and r["max_abs_dlogp"] == 0.0
    assert math.isnan(r["mean_dlogp"])
    r, o = _both(torch.tensor([0.0, 0.25, -0.25, 0.25]), torch.zeros(4), None)
    assert r["argmax_index"] == 1 and r["max_abs_dlogp"] == 0.25
    new = torch.zeros(9000)
    new[7000] = float("nan")
    new[8000] = 3.0
    r, o = _both(new, torch.zeros(9000), None)
    assert r["argmax_index"] == 7000 and math.isnan(r["max_abs_dlogp"]) and r["error_flags"] & 1
    r = rlk.dlogp_audit(torch.zeros(0, device=dev()), torch.zeros(0, device=dev()))
    assert r["active_count"] == 0 and r["argmax_index"] == -1


def test_pages_element_count_exact_and_reproducible():
    n = 9_400_614
    new, old, mask = wl.audit_inputs(n, 0)
    r, o = _both(new, old, mask)
    _check(r, o, new, old, mask)
    assert r["active_count"] == int(mask.sum())
    r2, _ = _both(new, old, mask)
    assert r == r2


def _block_slices(n, b):
    # the partition of pass 1: 4096-element slices dealt round-robin to min(slices, 608)
    # blocks; block b visits its slices in ascending order
    slices = -(-n // 4096)
    g = min(slices, 608)
    return list(range(b, slices, g))


def test_ties_across_the_slices_of_one_block():
    # At N = 5,000,000 (1221 slices) block 3 holds slices 3, 611 and 1219.  Equal largest |d|
    # in two slices of one block, in different float4 groups of the same thread, across two
    # blocks whose merge order is the opposite of their index order, and in the tail slice:
    # the lowest index must win each time.
    n = 5_000_000
    sl = _block_slices(n, 3)
    assert sl == [3, 611, 1219]
    new, old, mask = wl.audit_inputs(n, 9)
    mask[:] = 1
    cases = [
        (sl[1] * 4096 + 5, sl[0] * 4096 + 100),                      # block 3: slice 611 vs 3
        (sl[2] * 4096 + 1024 * 3 + 4 * 17, sl[0] * 4096 + 4 * 17),  # one thread: group 3 vs 0
        (612 * 4096 + 9, 5 * 4096 + 2000),        # block 4 (merged first) vs block 5
        (n - 3, n - 4096 * 2 - 7),                # the tail slice
    ]
    for later, earlier in cases:
        nw, od = new.clone(), old.clone()
        od[later] = od[earlier] = -1.0           # |d| = 0.75 exactly at both
        nw[later] = -0.25
        nw[earlier] = -1.75
        r, o = _both(nw, od, mask)
        _check(r, o, nw, od, mask)
        assert r["argmax_index"] == earlier, (later, earlier)


@pytest.mark.parametrize("n", [5003, 9_400_614])
def test_alignment_does_not_change_the_bits(n):
    # The same values placed at three alignments -- vector loads (all 16-byte aligned, or
    # the mask only 4-byte aligned) and element loads (values 4-byte aligned) -- go
    # through one arithmetic: the results are equal bit for bit.
    new, old, mask = wl.audit_inputs(n, 21)
    d = dev()
    out = []
    for off_v, off_m in ((0, 0), (4, 4), (1, 1)):
        nb = torch.zeros(n + 8, device=d)
        ob = torch.zeros(n + 8, device=d)
        mb = torch.zeros(n + 16, dtype=torch.uint8, device=d)
        nb[off_v:off_v + n] = new.to(d)
        ob[off_v:off_v + n] = old.to(d)
        mb[off_m:off_m + n] = mask.to(d)
        out.append(rlk.dlogp_audit(nb[off_v:off_v + n], ob[off_v:off_v + n], mb[off_m:off_m + n]))
    o = oracle.dlogp_audit(new.numpy(), old.numpy(), mask.numpy())
    _check(out[0], o, new, old, mask)
    for r in out[1:]:
        assert r == out[0] or all(
            (r[k] == out[0][k]) or (math.isnan(r[k]) and math.isnan(out[0][k])) for k in r)
