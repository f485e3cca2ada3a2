"""Seeded input recipes: shapes, length mixes, mask densities and determinism."""
import numpy as np
import torch

import workloads as wl


def test_tiny_recipe():
    w = wl.tiny_fwd(0)
    assert w.hidden.shape == (64, 128) and w.weight.shape == (1000, 128)
    assert w.hidden.dtype == torch.bfloat16 and w.targets.dtype == torch.int64
    assert w.n_active == 48
    assert all(int(w.mask[s * 32 + p]) == (1 if p < 24 else 0) for s in range(2) for p in range(32))
    assert int(w.targets.min()) >= 0 and int(w.targets.max()) < 1000
    w2 = wl.tiny_fwd(0)
    assert torch.equal(w.hidden.view(torch.int16), w2.hidden.view(torch.int16))
    assert abs(float(w.weight.float().std()) - 0.02) < 0.002


def test_packed_lengths():
    lens = wl.packed_lengths(8192, 8, 512, 2048, 0)
    assert sum(lens) == 8192 and len(lens) == 8 and all(512 <= x <= 2048 for x in lens)
    assert lens == wl.packed_lengths(8192, 8, 512, 2048, 0)


def test_normal_is_thread_count_independent(monkeypatch):
    a = wl.normal_bf16((3, (1 << 22) + 5), 3, wl.S_HIDDEN)
    monkeypatch.setattr(wl, "_threads", lambda: 1)
    b = wl.normal_bf16((3, (1 << 22) + 5), 3, wl.S_HIDDEN)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    x = a.float()
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01


def test_sampled_targets_follow_softmax():
    # with W = 0 the softmax is uniform; with one dominant logit the sample is that entry
    h = wl.normal_bf16((256, 16), 0, wl.S_HIDDEN)
    w = torch.zeros(50, 16, dtype=torch.bfloat16)
    y = wl.sample_targets(h, w, 0.7, 0)
    assert int(y.min()) >= 0 and int(y.max()) < 50 and len(set(y.tolist())) > 30
    w2 = torch.zeros(50, 16)
    w2[17] = 100.0 * torch.sign(h[0].float())
    y2 = wl.sample_targets(h[:1], w2.to(torch.bfloat16), 0.7, 0)
    assert int(y2[0]) == 17


def test_grpo_and_audit_inputs():
    noise, adv = wl.grpo_bwd_extras(100, [60, 40], 0)
    assert noise.shape == (100,) and len(set(adv[:60])) == 1 and len(set(adv[60:])) == 1
    new, old, mask = wl.audit_inputs(100000, 0)
    assert new.dtype == torch.float32 and mask.dtype == torch.uint8
    frac = float(mask.float().mean())
    assert 0.79 < frac < 0.81
    d = (new.double() - old.double()).numpy()
    assert abs(np.std(d) - 0.01) < 0.001


def test_sweep_lengths():
    lens = wl.sweep_lengths(0)
    assert len(lens) == 128 and all(128 <= x <= 4096 for x in lens)
