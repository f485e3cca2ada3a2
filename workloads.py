"""Seeded synthetic inputs shaped like the pages' GRPO workloads.

This module only draws random numbers and lays them out; it holds none of the
log-prob arithmetic.  The oracle (``oracle/``) and the CUDA library
(``rl_post_linear_gb300``) both consume what it returns, and neither imports
the other.  The one exception to "no arithmetic" is data preparation for the
Qwen-shaped forward, whose targets are drawn from the softmax of the logits
(see ``sample_targets``); both sides then receive the same target ids.

Recipes (page title and section in brackets):

* tiny_fwd -- N = 64 tokens (2 sequences x 32), H = 128, V = 1000, hidden
  ~ N(0,1), W ~ N(0, 0.02), targets uniform in [0, V), positions 24..31 of
  each sequence masked as padding, T = 1.0, seed 0.
* qwen_fwd -- the Qwen3-8B LM head ["RL-Kernel Roadmap (2026)", P1 and the
  v0.1.0 announcement's Qwen3-8B GRPO runs]: H = 4096, V = 151936, N = 8192
  tokens packed from 8 sequences with lengths uniform in 512..2048 summing to
  8192, all active, T = 0.7, targets sampled from the softmax of the logits.
* deepseek_fwd -- a DeepSeek-style large head: H = 7168, V = 129280,
  N = 16384 (32 x 512), W ~ N(0, 0.015), 20% of tokens masked (i.i.d.),
  T = 1.0, targets uniform.
* grpo_bwd_extras -- the GRPO clipped-ratio backward inputs: old logp noise
  ~ N(0, 0.01) per token, advantages ~ N(0, 1) per sequence, eps = 0.2.
* sweep_samples -- the batch-invariance sweep ["RL-Kernel integration roadmap
  for vime", Consistency Contract]: GRPO groups of 8 responses for 16
  prompts, response lengths uniform in 128..4096, each sample's hidden rows
  and targets drawn from its own seed.
* audit_inputs -- dlogp audit vectors: d ~ N(0, 0.01), mask Bernoulli(0.8).

Normal draws use numpy's Philox bit generator on fixed-size chunks (seeded
through ``SeedSequence([seed, stream, chunk])``), so the values do not depend
on the number of host threads; fp32 values are rounded to bf16 with
round-to-nearest-even by torch.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

_CHUNK = 1 << 22

# stream ids keep every drawn tensor independent of the others
S_HIDDEN, S_WEIGHT, S_TARGET, S_MASK, S_LENGTHS, S_NOISE, S_ADV, S_SWEEP, S_AUDIT, S_PAD = range(1, 11)


def _threads():
    return max(1, len(os.sched_getaffinity(0)))


def _gen(seed, stream, idx=0):
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, stream, idx])))


def normal_f32(n, seed, stream, std=1.0):
    """n float32 draws from N(0, std^2)."""
    out = np.empty(n, np.float32)
    nch = (n + _CHUNK - 1) // _CHUNK

    def work(i):
        a, b = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        _gen(seed, stream, i).standard_normal(out=out[a:b], dtype=np.float32)
        if std != 1.0:
            out[a:b] *= np.float32(std)

    if nch:
        with ThreadPoolExecutor(min(nch, _threads())) as ex:
            list(ex.map(work, range(nch)))
    return out


def normal_bf16(shape, seed, stream, std=1.0):
    """bf16 tensor of the given shape: fp32 N(0, std^2) draws rounded to nearest even."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(n, dtype=torch.bfloat16)
    nch = (n + _CHUNK - 1) // _CHUNK

    def work(i):
        a, b = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        x = _gen(seed, stream, i).standard_normal(b - a, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[a:b] = torch.from_numpy(x).to(torch.bfloat16)

    if nch:
        with ThreadPoolExecutor(min(nch, _threads())) as ex:
            list(ex.map(work, range(nch)))
    return out.view(*shape)


@dataclass
class Workload:
    name: str
    hidden: torch.Tensor          # [N, H] bf16 (CPU)
    weight: torch.Tensor          # [V, H] bf16 (CPU)
    targets: torch.Tensor         # [N] int64
    mask: torch.Tensor            # [N] uint8, nonzero = active
    temperature: float
    seq_lens: list = field(default_factory=list)

    @property
    def n(self):
        return self.hidden.shape[0]

    @property
    def h(self):
        return self.hidden.shape[1]

    @property
    def v(self):
        return self.weight.shape[0]

    @property
    def n_active(self):
        return int(self.mask.sum())


def uniform_targets(n, vocab, seed):
    return torch.from_numpy(_gen(seed, S_TARGET).integers(0, vocab, size=n, dtype=np.int64))


def packed_lengths(total, count, lo, hi, seed):
    """count lengths in [lo, hi] summing to total: draw the first count-1 uniformly and
    redraw until the last one also lands in [lo, hi]."""
    g = _gen(seed, S_LENGTHS)
    for _ in range(100000):
        first = g.integers(lo, hi + 1, size=count - 1)
        last = total - int(first.sum())
        if lo <= last <= hi:
            return [int(x) for x in first] + [last]
    raise RuntimeError("no admissible length draw")


def sample_targets(hidden, weight, temperature, seed, rows_per_block=512):
    """Targets drawn from softmax(h W^T / T) by inverse-CDF sampling, one uniform per token.

    Data preparation only: logits are formed in fp32 on the host from the same bf16
    inputs, block by block, and never stored.
    """
    n = hidden.shape[0]
    u = _gen(seed, S_TARGET).random(n)
    wf = weight.float()
    out = torch.empty(n, dtype=torch.int64)
    for a in range(0, n, rows_per_block):
        b = min(n, a + rows_per_block)
        z = (hidden[a:b].float() @ wf.T) / temperature
        p = torch.softmax(z.double(), dim=1)
        c = torch.cumsum(p, dim=1)
        uu = torch.from_numpy(u[a:b]).unsqueeze(1) * c[:, -1:]
        idx = torch.searchsorted(c, uu).squeeze(1)
        out[a:b] = idx.clamp_(max=weight.shape[0] - 1)
    return out


def tiny_fwd(seed=0):
    n_seq, seq_len, hdim, vocab = 2, 32, 128, 1000
    n = n_seq * seq_len
    hidden = normal_bf16((n, hdim), seed, S_HIDDEN)
    weight = normal_bf16((vocab, hdim), seed, S_WEIGHT, std=0.02)
    targets = uniform_targets(n, vocab, seed)
    mask = torch.ones(n, dtype=torch.uint8)
    for s in range(n_seq):
        mask[s * seq_len + 24:(s + 1) * seq_len] = 0       # last 25% of each row is padding
    return Workload("tiny_fwd N=64 H=128 V=1000", hidden, weight, targets, mask, 1.0,
                    [seq_len] * n_seq)


QWEN_H, QWEN_V, QWEN_N = 4096, 151936, 8192
DEEPSEEK_H, DEEPSEEK_V, DEEPSEEK_N = 7168, 129280, 16384


def qwen_fwd(seed=0, n_tokens=QWEN_N, sample=True):
    lens = packed_lengths(n_tokens, 8, 512, 2048, seed) if n_tokens == QWEN_N else [n_tokens]
    hidden = normal_bf16((n_tokens, QWEN_H), seed, S_HIDDEN)
    weight = normal_bf16((QWEN_V, QWEN_H), seed, S_WEIGHT, std=0.02)
    if sample:
        targets = sample_targets(hidden, weight, 0.7, seed)
    else:
        targets = uniform_targets(n_tokens, QWEN_V, seed)
    mask = torch.ones(n_tokens, dtype=torch.uint8)
    return Workload("qwen3-8b lm-head fwd N=%d H=4096 V=151936 T=0.7" % n_tokens, hidden, weight,
                    targets, mask, 0.7, lens)


def deepseek_fwd(seed=0):
    hidden = normal_bf16((DEEPSEEK_N, DEEPSEEK_H), seed, S_HIDDEN)
    weight = normal_bf16((DEEPSEEK_V, DEEPSEEK_H), seed, S_WEIGHT, std=0.015)
    targets = uniform_targets(DEEPSEEK_N, DEEPSEEK_V, seed)
    mask = torch.from_numpy((_gen(seed, S_MASK).random(DEEPSEEK_N) >= 0.2).astype(np.uint8))
    return Workload("deepseek-style fwd N=16384 H=7168 V=129280 T=1.0", hidden, weight, targets,
                    mask, 1.0, [512] * 32)


def grpo_bwd_extras(n, seq_lens, seed=0):
    """(old-logp noise [N] float64 ~ N(0, 0.01^2), advantages [N] float64 constant per sequence)."""
    noise = _gen(seed, S_NOISE).normal(0.0, 0.01, size=n)
    adv_seq = _gen(seed, S_ADV).normal(0.0, 1.0, size=len(seq_lens))
    adv = np.repeat(adv_seq, seq_lens)
    assert adv.shape[0] == n
    return noise, adv


GRPO_EPS = 0.2


def sweep_lengths(seed=0, prompts=16, group=8, lo=128, hi=4096):
    return [int(x) for x in _gen(seed, S_SWEEP).integers(lo, hi + 1, size=prompts * group)]


def sweep_sample(i, length, hdim, vocab, seed=0):
    """hidden rows [length, H] bf16 and targets [length] of sample i, from the sample's own seed."""
    s = seed * 1000003 + i + 1
    return normal_bf16((length, hdim), s, S_HIDDEN), uniform_targets(length, vocab, s)


def padding_rows(count, hdim, seed):
    """finite random padding rows (the backward needs finite padding)."""
    return normal_bf16((count, hdim), seed, S_PAD)


def permutation(n, seed, stream=S_SWEEP):
    return [int(x) for x in _gen(seed, stream, 7).permutation(n)]


def audit_inputs(n, seed=0):
    """(logp_new, logp_old) float32 [N] and mask uint8 [N]: old ~ -Exp(1), new = old + d,
    d ~ N(0, 0.01^2), mask Bernoulli(0.8)."""
    g = _gen(seed, S_AUDIT)
    old = (-g.exponential(1.0, size=n)).astype(np.float32)
    d = normal_f32(n, seed, S_AUDIT, std=0.01)
    new = (old + d).astype(np.float32)
    mask = (g.random(n) < 0.8).astype(np.uint8)
    return torch.from_numpy(new), torch.from_numpy(old), torch.from_numpy(mask)


def describe(w: Workload):
    return {"workload": w.name, "n_tokens": w.n, "n_active": w.n_active, "hidden": w.h,
            "vocab": w.v, "temperature": w.temperature}
