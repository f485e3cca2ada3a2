"""logp from existing logits ("RL-Kernel integration roadmap for vime", logp
Reference Scoring): parity with the oracle, bitwise equality of dense and
indexed rows and across batches, and agreement with the fused linear path on
the same inputs."""
import numpy as np
import pytest
import torch

import oracle
import rl_post_linear_gb300 as rlk
import workloads as wl
from helpers import LOGP_ATOL, dev, same_bits

pytestmark = pytest.mark.gpu


def _case(n, v, seed, dtype, stride=None):
    g = np.random.default_rng(seed)
    z = torch.from_numpy((g.standard_normal((n, stride or v)) * 2.0).astype(np.float32))
    z = z.to(dtype)
    y = torch.from_numpy(g.integers(0, v, n))
    m = torch.from_numpy((g.random(n) < 0.85).astype(np.uint8))
    return z, y, m


@pytest.mark.parametrize("n,v,dtype,stride,T", [(64, 1000, torch.float32, None, 1.0),
                                                (33, 151936, torch.float32, None, 0.7),
                                                (50, 4097, torch.bfloat16, None, 0.5),
                                                (17, 1001, torch.float32, 1003, 1.3),
                                                (20, 3000, torch.bfloat16, 3008, 0.9)])
def test_parity(n, v, dtype, stride, T):
    z, y, m = _case(n, v, n + v, dtype, stride)
    d = dev()
    zd = z.to(d)[:, :v] if stride else z.to(d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    logp, lse = rlk.logp_from_logits(zd, y.to(d), m.to(d), T, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    z64 = z[:, :v].double().numpy() if dtype == torch.float32 else z[:, :v].float().double().numpy()
    lp_o, lse_o = oracle.logp_from_logits(z64, y.numpy(), m.numpy(), T)
    act = m.numpy() > 0
    dl = np.abs(logp.cpu().double().numpy() - lp_o)[act]
    assert dl.max() <= LOGP_ATOL
    assert np.abs(lse.cpu().double().numpy() - lse_o)[act].max() <= LOGP_ATOL
    assert np.all(logp.cpu().numpy()[~act] == 0)
    print("logits parity n=%d v=%d %s: max |dlogp| %.3e" % (n, v, dtype, dl.max()))


def test_dense_vs_indexed_and_batch_invariance():
    z, y, m = _case(200, 5000, 3, torch.float32)
    d = dev()
    zd, yd, md = z.to(d), y.to(d), m.to(d)
    dense, dlse = rlk.logp_from_logits(zd, yd, md, 0.7)
    rows = torch.tensor([199, 0, 57, 57, 3, 120], dtype=torch.int64, device=d)
    idx, ilse = rlk.logp_from_logits(zd, yd, md, 0.7, rows=rows)
    assert same_bits(idx.cpu(), dense[rows].cpu()) and same_bits(ilse.cpu(), dlse[rows].cpu())
    part, plse = rlk.logp_from_logits(zd[50:90], yd[50:90], md[50:90], 0.7)
    assert same_bits(part.cpu(), dense[50:90].cpu()) and same_bits(plse.cpu(), dlse[50:90].cpu())


def test_agrees_with_fused_linear_path():
    d = dev()
    n, h, v = 128, 512, 20000
    hid = wl.normal_bf16((n, h), 5, wl.S_HIDDEN).to(d)
    w = wl.normal_bf16((v, h), 5, wl.S_WEIGHT, std=0.05).to(d)
    y = wl.uniform_targets(n, v, 5).to(d)
    fused, flse = rlk.linear_logp_fwd(hid, w, y, None, 0.7)
    logits = hid.float() @ w.float().T          # exact products, fp32 sums
    lp, lse = rlk.logp_from_logits(logits, y, None, 0.7)
    assert float((lp - fused).abs().max()) < 1e-4 and float((lse - flse).abs().max()) < 1e-4


def test_bad_row_index_is_flagged():
    z, y, m = _case(10, 100, 9, torch.float32)
    d = dev()
    err = torch.zeros(1, dtype=torch.int32, device=d)
    rows = torch.tensor([0, 10, -1, 5], dtype=torch.int64, device=d)
    lp, _ = rlk.logp_from_logits(z.to(d), y.to(d), None, 1.0, rows=rows, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & rlk.RLK_DEVERR_ROW_RANGE
    assert torch.isnan(lp[1]).item() and torch.isnan(lp[2]).item() and torch.isfinite(lp[0]).item()
