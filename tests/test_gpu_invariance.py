"""Batch-invariance sweep: a sample's logp, lse and dhidden are bitwise equal
whatever batch it is scored in ("RL-Kernel integration roadmap for vime",
Consistency Contract: the same sample scored alone, in a different batch,
padded differently, packed in a different order or in another microbatch must
not change; "RL-Kernel Roadmap (2026)", P0.2 batch-invariant deterministic
logprob).

GRPO groups of 8 responses for 16 prompts (128 samples), response lengths
uniform in 128..4096, H = 4096, V = 151936, T = 0.7.  Each sample's hidden rows,
targets and (fixed, per-sample) upstream gradient come from its own seed.
Layouts: every sample alone; every batch of 2 / 8 / 32 / 128 samples of a
seeded random order (all 64 pairs, 16 eights, 4 thirty-twos, 1 full batch, so
each sample is scored in four batches), each packed back to back, right-padded
and left-padded to the longest sample with finite random padding rows
(masked).  dweight sums over the batch,
so it is checked for run-to-run bitwise reproducibility instead.
"""
import numpy as np
import pytest
import torch

import rl_post_linear_gb300 as rlk
import workloads as wl
from helpers import dev

pytestmark = pytest.mark.gpu

H, V, T = wl.QWEN_H, wl.QWEN_V, 0.7


@pytest.fixture(scope="module")
def sweep():
    d = dev()
    lens = wl.sweep_lengths(0)
    samples = []
    for i, ln in enumerate(lens):
        h, y = wl.sweep_sample(i, ln, H, V, 0)
        g = torch.from_numpy(np.random.default_rng(10_000 + i).standard_normal(ln) * 1e-3).float()
        samples.append((h.to(d), y.to(d), g.to(d)))
    weight = wl.normal_bf16((V, H), 0, wl.S_WEIGHT, std=0.02).to(d)
    pad_pool = wl.padding_rows(4096 + 127, H, 99).to(d)
    return lens, samples, weight, pad_pool


def _score(weight, h, y, m, g):
    err = torch.zeros(1, dtype=torch.int32, device=h.device)
    logp, lse = rlk.linear_logp_fwd(h, weight, y, m, T, err)
    dh, dw = rlk.linear_logp_bwd(h, weight, y, m, g, lse, T, err)
    assert int(err.item()) == 0
    return logp, lse, dh, dw


def _layout(samples, order, mode, pad_pool):
    """Concatenate the samples in `order`: packed, or padded right/left to the longest."""
    d = samples[0][0].device
    longest = max(samples[i][0].shape[0] for i in order)
    hs, ys, ms, gs, where = [], [], [], [], []
    row = 0
    for j, i in enumerate(order):
        h, y, g = samples[i]
        ln = h.shape[0]
        pad = 0 if mode == "packed" else longest - ln
        ph = pad_pool[j % 128: j % 128 + pad]
        py = torch.zeros(pad, dtype=torch.int64, device=d)
        pm = torch.zeros(pad, dtype=torch.uint8, device=d)
        pg = torch.zeros(pad, dtype=torch.float32, device=d)
        ones = torch.ones(ln, dtype=torch.uint8, device=d)
        parts = [(h, y, ones, g), (ph, py, pm, pg)]
        if mode == "left":
            parts.reverse()
        for a, b, c, e in parts:
            hs.append(a)
            ys.append(b)
            ms.append(c)
            gs.append(e)
        start = row + (pad if mode == "left" else 0)
        where.append((i, start, ln))
        row += ln + pad
    return torch.cat(hs), torch.cat(ys), torch.cat(ms), torch.cat(gs), where


def test_sweep_bitwise(sweep):
    lens, samples, weight, pad_pool = sweep
    ref = []
    for h, y, g in samples:
        logp, lse, dh, _ = _score(weight, h, y, torch.ones_like(y, dtype=torch.uint8), g)
        ref.append((logp.clone(), lse.clone(), dh.clone()))
    mismatches = 0
    checked = 0
    rng = np.random.default_rng(0)
    for bs in (2, 8, 32, 128):
        order_all = [int(i) for i in rng.permutation(len(samples))]
        for mode in ("packed", "right", "left"):
            for b0 in range(0, len(samples), bs):
                order = order_all[b0:b0 + bs]
                h, y, m, g, where = _layout(samples, order, mode, pad_pool)
                logp, lse, dh, _ = _score(weight, h, y, m, g)
                for i, start, ln in where:
                    r = ref[i]
                    sl = slice(start, start + ln)
                    mismatches += int((logp[sl].view(torch.int32) != r[0].view(torch.int32)).sum())
                    mismatches += int((lse[sl].view(torch.int32) != r[1].view(torch.int32)).sum())
                    mismatches += int((dh[sl].view(torch.int16) != r[2].view(torch.int16)).sum())
                    checked += ln
    print("batch-invariance sweep: %d sample-rows compared, %d mismatching elements"
          % (checked, mismatches))
    assert mismatches == 0


def test_dweight_run_to_run(sweep):
    lens, samples, weight, pad_pool = sweep
    order = list(range(16))
    h, y, m, g, _ = _layout(samples, order, "packed", pad_pool)
    _, _, _, dw1 = _score(weight, h, y, m, g)
    dw1 = dw1.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _, _, _, dw2 = _score(weight, h, y, m, g)
    torch.cuda.synchronize()
    assert torch.equal(dw1.view(torch.int16), dw2.view(torch.int16))
