"""Parity at the pages' full workload shapes, in the launch configuration the
benchmark times.

* Qwen3-8B-shaped forward (N = 8192, H = 4096, V = 151936, T = 0.7, sampled
  targets): 256 sampled tokens -- the first and last token of every packed
  sequence, both sides of every 128-row tile edge in range, and seeded random
  ones -- against the oracle, token by token.
* Qwen-shaped GRPO backward: the whole dh and dW tensors against the oracle at
  N = 256 with the full H and V (four 64-token K blocks in the dW GEMM); at
  N = 8192, 16 sampled dh rows against the oracle and, for dW, the
  softmax-gradient identity sum_v dW_v = 0 (each column sum must vanish up to
  the bf16 output rounding).
* Entropy and full-vocabulary KL backwards at the Qwen shape (N = 8192):
  sampled dh rows against the oracle and the same column-sum identity of dW
  (the entropy and both KL gradients also sum to zero over the vocabulary).
* DeepSeek-shaped forward (N = 16384, H = 7168, V = 129280, 20% masked):
  128 sampled tokens.
* DeepSeek-shaped backward (the same masked batch, compacted to its active
  rows): 16 sampled active dh rows against the oracle, exact zeros on the
  inactive rows, and the column sums of dW.
* Audit at N = 2^26.
"""
import numpy as np
import pytest
import torch

import oracle
import rl_post_linear_gb300 as rlk
import workloads as wl
from helpers import GRAD_REL_L2, LOGP_ATOL, dev, f64, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qwen():
    w = wl.qwen_fwd(0)
    w64 = oracle.bf16_bits_to_f64(w.weight)
    return w, w64


def _sample_rows(w, count, seed):
    rows = set()
    start = 0
    for ln in w.seq_lens:
        rows.update((start, start + ln - 1))
        start += ln
    for edge in range(128, w.n, 128 * 7):
        rows.update((edge - 1, edge))
    rows.update((0, w.n - 1))
    rng = np.random.default_rng(seed)
    while len(rows) < count:
        rows.add(int(rng.integers(0, w.n)))
    return np.array(sorted(rows)[:max(count, len(rows))], dtype=np.int64)


def test_qwen_forward_sampled(qwen):
    w, w64 = qwen
    d = dev()
    err = torch.zeros(1, dtype=torch.int32, device=d)
    logp, lse = rlk.linear_logp_fwd(w.hidden.to(d), w.weight.to(d), w.targets.to(d),
                                    w.mask.to(d), w.temperature, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = _sample_rows(w, 256, 1)
    lp_o, lse_o = oracle.linear_logp_fwd_parallel(f64(w.hidden[rows]), w64,
                                                  w.targets[rows].numpy(), None, w.temperature)
    dl = np.abs(logp.cpu().double().numpy()[rows] - lp_o)
    dz = np.abs(lse.cpu().double().numpy()[rows] - lse_o)
    print("qwen fwd: %d sampled tokens, max |dlogp| %.3e, max |dlse| %.3e" % (len(rows), dl.max(),
                                                                               dz.max()))
    assert dl.max() <= LOGP_ATOL and dz.max() <= LOGP_ATOL
    assert np.all(logp.cpu().numpy() <= 1e-6)


def _grpo_g(logp_o, w, seed, rows):
    noise, adv = wl.grpo_bwd_extras(w.n, w.seq_lens, seed)
    old = logp_o + noise[rows]
    _, g = oracle.grpo_clip_grad(logp_o, old, adv[rows], w.mask[rows].numpy(), wl.GRPO_EPS)
    return g


def test_qwen_backward_full_tensors_reduced_n(qwen):
    w, w64 = qwen
    n = 256
    rows = np.arange(n)
    h = w.hidden[:n]
    y = w.targets[:n]
    m = w.mask[:n]
    h64 = f64(h)
    lp_o, lse_o = oracle.linear_logp_fwd_parallel(h64, w64, y.numpy(), m.numpy(), w.temperature)
    g = _grpo_g(lp_o, w, 0, rows)
    d = dev()
    err = torch.zeros(1, dtype=torch.int32, device=d)
    hd, wd, yd, md = h.to(d), w.weight.to(d), y.to(d), m.to(d)
    _, lse = rlk.linear_logp_fwd(hd, wd, yd, md, w.temperature, err)
    dh, dw = rlk.linear_logp_bwd(hd, wd, yd, md, torch.tensor(g, dtype=torch.float32, device=d),
                                 lse, w.temperature, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    dh_o = oracle.linear_logp_bwd_dh_parallel(h64, w64, y.numpy(), m.numpy(), g, lse_o,
                                              w.temperature)
    e_dh = rel_l2(dh, dh_o)
    dw_gpu = f64(dw)
    acc = {"num": 0.0, "den": 0.0, "num_r": 0.0}
    import threading
    lock = threading.Lock()

    def consume(v0, blk):
        gb = dw_gpu[v0:v0 + blk.shape[0]]
        rounded = torch.from_numpy(blk).float().to(torch.bfloat16).double().numpy()
        with lock:
            acc["num"] += float(np.sum((gb - blk) ** 2))
            acc["den"] += float(np.sum(blk ** 2))
            acc["num_r"] += float(np.sum((gb - rounded) ** 2))

    oracle.linear_logp_bwd_dw_blocks(h64, w64, y.numpy(), m.numpy(), g, lse_o, w.temperature, 0,
                                     w.v, consume, rows_per_block=512)
    e_dw = (acc["num"] / acc["den"]) ** 0.5
    e_dw_r = (acc["num_r"] / acc["den"]) ** 0.5
    print("qwen bwd N=%d: rel-L2 dh %.3e dw %.3e (dw vs bf16-rounded oracle %.3e)"
          % (n, e_dh, e_dw, e_dw_r))
    assert e_dh <= GRAD_REL_L2 and e_dw <= GRAD_REL_L2


def test_qwen_backward_full_size(qwen):
    w, w64 = qwen
    d = dev()
    err = torch.zeros(1, dtype=torch.int32, device=d)
    hd, wd, yd, md = w.hidden.to(d), w.weight.to(d), w.targets.to(d), w.mask.to(d)
    # upstream gradient: GRPO clipped ratio with per-token coefficients from the oracle at the
    # sampled rows; every other row gets a seeded gradient of the same scale
    rows = _sample_rows(w, 16, 2)
    lp_o, lse_o = oracle.linear_logp_fwd_parallel(f64(w.hidden[rows]), w64,
                                                  w.targets[rows].numpy(), None, w.temperature)
    g = np.random.default_rng(5).standard_normal(w.n) / w.n
    g[rows] = _grpo_g(lp_o, w, 0, rows) * len(rows) / w.n
    gd = torch.tensor(g, dtype=torch.float32, device=d)
    _, lse = rlk.linear_logp_fwd(hd, wd, yd, md, w.temperature, err)
    dh, dw = rlk.linear_logp_bwd(hd, wd, yd, md, gd, lse, w.temperature, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    g32 = gd.cpu().double().numpy()
    dh_o = oracle.linear_logp_bwd_dh_parallel(f64(w.hidden[rows]), w64, w.targets[rows].numpy(),
                                              None, g32[rows], lse_o, w.temperature)
    e = rel_l2(dh.cpu()[rows], dh_o)
    # softmax-gradient identity: every column of dW sums to zero
    col = dw.double().sum(dim=0)
    rms = dw.double().pow(2).sum(dim=0).sqrt()
    worst = float((col.abs() / rms).max())
    print("qwen bwd N=8192: sampled dh rel-L2 %.3e; max |col sum| / col norm %.3e" % (e, worst))
    assert e <= GRAD_REL_L2
    assert worst <= 8 * 2.0 ** -8


def test_deepseek_forward_sampled():
    w = wl.deepseek_fwd(0)
    d = dev()
    err = torch.zeros(1, dtype=torch.int32, device=d)
    logp, lse = rlk.linear_logp_fwd(w.hidden.to(d), w.weight.to(d), w.targets.to(d),
                                    w.mask.to(d), w.temperature, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = _sample_rows(w, 128, 3)
    rows = rows[w.mask.numpy()[rows] > 0]
    lp_o, lse_o = oracle.linear_logp_fwd_parallel(f64(w.hidden[rows]), f64(w.weight),
                                                  w.targets[rows].numpy(), None, w.temperature)
    dl = np.abs(logp.cpu().double().numpy()[rows] - lp_o)
    print("deepseek fwd: %d sampled tokens, max |dlogp| %.3e" % (len(rows), dl.max()))
    assert dl.max() <= LOGP_ATOL
    inactive = w.mask.numpy() == 0
    assert np.all(logp.cpu().numpy()[inactive] == 0.0)


def test_deepseek_backward_sampled():
    w = wl.deepseek_fwd(0)
    d = dev()
    err = torch.zeros(1, dtype=torch.int32, device=d)
    hd, wd, yd, md = w.hidden.to(d), w.weight.to(d), w.targets.to(d), w.mask.to(d)
    act = w.mask.numpy() > 0
    g = np.random.default_rng(5).standard_normal(w.n) / w.n_active
    g[~act] = 0.0
    gd = torch.tensor(g, dtype=torch.float32, device=d)
    _, lse = rlk.linear_logp_fwd(hd, wd, yd, md, w.temperature, err)
    dh, dw = rlk.linear_logp_bwd(hd, wd, yd, md, gd, lse, w.temperature, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = _sample_rows(w, 24, 4)
    rows = rows[act[rows]][:16]
    w64 = f64(w.weight)
    h64 = f64(w.hidden[rows])
    _, lse_o = oracle.linear_logp_fwd_parallel(h64, w64, w.targets[rows].numpy(), None,
                                               w.temperature)
    g32 = gd.cpu().double().numpy()
    dh_o = oracle.linear_logp_bwd_dh_parallel(h64, w64, w.targets[rows].numpy(), None,
                                              g32[rows], lse_o, w.temperature)
    dh_c = dh.cpu()
    e = rel_l2(dh_c[rows], dh_o)
    assert torch.all(dh_c[torch.from_numpy(~act)].float() == 0)
    col = dw.double().sum(dim=0)
    rms = dw.double().pow(2).sum(dim=0).sqrt()
    worst = float((col.abs() / rms).max())
    print("deepseek bwd: %d sampled dh rows rel-L2 %.3e; max |col sum| / col norm %.3e"
          % (len(rows), e, worst))
    assert e <= GRAD_REL_L2
    assert worst <= 8 * 2.0 ** -8


def test_audit_two_to_the_26():
    n = 1 << 26
    new, old, mask = wl.audit_inputs(n, 1)
    d = dev()
    r = rlk.dlogp_audit(new.to(d), old.to(d), mask.to(d))
    o = oracle.dlogp_audit(new.numpy(), old.numpy(), mask.numpy())
    assert r["active_count"] == o["active_count"] == int(mask.sum())
    assert r["argmax_index"] == o["argmax_index"]
    assert r["max_abs_dlogp"] == np.float32(o["max_abs_dlogp"])
    assert abs(r["approx_kl"] - o["approx_kl"]) <= 1e-6 * o["approx_kl"]


def test_qwen_entropy_and_kl_sampled(qwen):
    # the next rows at the shape the benchmark times them: entropy of the policy, and the
    # full-vocabulary KL against a reference head of the same shape, on sampled tokens
    w, w64 = qwen
    d = dev()
    hd, wd, yd, md = w.hidden.to(d), w.weight.to(d), w.targets.to(d), w.mask.to(d)
    _, _, ent = rlk.linear_logp_entropy_fwd(hd, wd, yd, md, w.temperature)
    rows = _sample_rows(w, 24, 7)
    _, _, ent_o = oracle.linear_logp_entropy_fwd_parallel(f64(w.hidden[rows]), w64,
                                                          w.targets[rows].numpy(), None,
                                                          w.temperature)
    de = np.abs(ent.cpu().double().numpy()[rows] - ent_o)
    hr = wl.normal_bf16((w.n, w.h), 1, wl.S_HIDDEN)
    wr = wl.normal_bf16((w.v, w.h), 1, wl.S_WEIGHT, std=0.02)
    kl, kr, lse, lse_r, _ = rlk.linear_kl_fwd(hd, wd, hr.to(d), wr.to(d), md, w.temperature,
                                              1.0)
    rows = rows[:12]
    o = oracle.linear_kl_fwd_parallel(f64(w.hidden[rows]), w64, f64(hr[rows]),
                                      oracle.bf16_bits_to_f64(wr), None, w.temperature, 1.0)
    dk = [np.abs(x.cpu().double().numpy()[rows] - e).max() for x, e in zip((kl, kr, lse, lse_r), o)]
    print("qwen entropy: max |dH| %.3e (H ~ %.2f); KL ~ %.3f: max |d| kl %.2e rev %.2e lse %.2e "
          "%.2e" % (de.max(), ent_o.mean(), o[0].mean(), *dk))
    assert de.max() <= LOGP_ATOL and max(dk) <= LOGP_ATOL


def _column_identity(dw):
    # sum_v dW_v = 0 for a gradient whose rows sum to zero over the vocabulary
    col = dw.double().sum(dim=0)
    rms = dw.double().pow(2).sum(dim=0).sqrt()
    return float((col.abs() / rms).max())


def test_qwen_entropy_backward_sampled(qwen):
    w, w64 = qwen
    d = dev()
    err = torch.zeros(1, dtype=torch.int32, device=d)
    hd, wd, yd, md = w.hidden.to(d), w.weight.to(d), w.targets.to(d), w.mask.to(d)
    rng = np.random.default_rng(11)
    gd = torch.tensor(rng.standard_normal(w.n) / w.n, dtype=torch.float32, device=d)
    ghd = torch.tensor(rng.standard_normal(w.n) / w.n, dtype=torch.float32, device=d)
    _, lse, ent = rlk.linear_logp_entropy_fwd(hd, wd, yd, md, w.temperature, err)
    dh, dw = rlk.linear_logp_entropy_bwd(hd, wd, yd, md, gd, ghd, lse, ent, w.temperature, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = _sample_rows(w, 16, 12)
    h64 = f64(w.hidden[rows])
    y = w.targets[rows].numpy()
    _, lse_o, ent_o = oracle.linear_logp_entropy_fwd_parallel(h64, w64, y, None, w.temperature)
    dh_o = oracle.linear_logp_entropy_bwd_dh_parallel(
        h64, w64, y, None, gd.cpu().double().numpy()[rows], ghd.cpu().double().numpy()[rows],
        lse_o, ent_o, w.temperature)
    e = rel_l2(dh.cpu()[rows], dh_o)
    worst = _column_identity(dw)
    print("qwen entropy bwd N=8192: sampled dh rel-L2 %.3e; max |col sum| / col norm %.3e"
          % (e, worst))
    assert e <= GRAD_REL_L2
    assert worst <= 8 * 2.0 ** -8


def test_qwen_kl_backward_sampled(qwen):
    w, w64 = qwen
    d = dev()
    err = torch.zeros(1, dtype=torch.int32, device=d)
    hd, wd, md = w.hidden.to(d), w.weight.to(d), w.mask.to(d)
    hr = wl.normal_bf16((w.n, w.h), 1, wl.S_HIDDEN)
    wr = wl.normal_bf16((w.v, w.h), 1, wl.S_WEIGHT, std=0.02)
    hrd, wrd = hr.to(d), wr.to(d)
    rng = np.random.default_rng(13)
    gd = torch.tensor(rng.standard_normal(w.n) / w.n, dtype=torch.float32, device=d)
    grd = torch.tensor(rng.standard_normal(w.n) / w.n, dtype=torch.float32, device=d)
    kl, _, lse, lse_r, _ = rlk.linear_kl_fwd(hd, wd, hrd, wrd, md, w.temperature, 1.0)
    dh, dw = rlk.linear_kl_bwd(hd, wd, hrd, wrd, md, gd, grd, lse, lse_r, kl, w.temperature, 1.0,
                               err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = _sample_rows(w, 12, 14)
    h64, hr64 = f64(w.hidden[rows]), f64(hr[rows])
    wr64 = oracle.bf16_bits_to_f64(wr)
    kl_o, _, lse_o, lse_ro = oracle.linear_kl_fwd_parallel(h64, w64, hr64, wr64, None,
                                                           w.temperature, 1.0)
    dh_o = oracle.linear_kl_bwd_dh_parallel(h64, w64, hr64, wr64, None,
                                            gd.cpu().double().numpy()[rows],
                                            grd.cpu().double().numpy()[rows], lse_o, lse_ro,
                                            kl_o, w.temperature, 1.0)
    e = rel_l2(dh.cpu()[rows], dh_o)
    worst = _column_identity(dw)
    print("qwen kl bwd N=8192: sampled dh rel-L2 %.3e; max |col sum| / col norm %.3e"
          % (e, worst))
    assert e <= GRAD_REL_L2
    assert worst <= 8 * 2.0 ** -8
