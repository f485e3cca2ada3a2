"""A batch eight times the benchmark's: N = 65536 tokens at the Qwen3-8B head
shape (H = 4096, V = 151936), 10% of rows masked.

At this size the backward's dS chunk is 4.3 GB (more than 2^31 elements), the
dW GEMM runs K = 65536 in one pass, the target list is sorted in 32 tiles and
the forward walks 16 raster groups of token tiles.  Checked: sampled logp and
dh rows against the oracle, the dW column-sum identity, dW run to run, and
bitwise equality of logp / lse / dh rows with the same rows scored in a batch
of 300 ("RL-Kernel integration roadmap for vime", Consistency Contract).
"""
import numpy as np
import pytest
import torch

import oracle
import rl_post_linear_gb300 as rlk
import workloads as wl
from helpers import GRAD_REL_L2, LOGP_ATOL, dev, f64, rel_l2, same_bits

pytestmark = pytest.mark.gpu

N, H, V, T = 65536, wl.QWEN_H, wl.QWEN_V, 0.7


@pytest.fixture(scope="module")
def big():
    hidden = wl.normal_bf16((N, H), 11, wl.S_HIDDEN)
    weight = wl.normal_bf16((V, H), 11, wl.S_WEIGHT, std=0.02)
    targets = wl.uniform_targets(N, V, 11)
    rng = np.random.default_rng(11)
    mask = torch.from_numpy((rng.random(N) >= 0.1).astype(np.uint8))
    grad = rng.standard_normal(N) / N
    grad[mask.numpy() == 0] = 0.0
    d = dev()
    hd, wd, yd, md = hidden.to(d), weight.to(d), targets.to(d), mask.to(d)
    gd = torch.tensor(grad, dtype=torch.float32, device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    logp, lse = rlk.linear_logp_fwd(hd, wd, yd, md, T, err)
    dh, dw = rlk.linear_logp_bwd(hd, wd, yd, md, gd, lse, T, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # rows to sample: both sides of the first and last tile and sort-tile edges, plus random
    rows = {0, 127, 128, 2047, 2048, N - 129, N - 128, N - 1}
    rows.update(int(r) for r in rng.integers(0, N, 24))
    rows = np.array(sorted(r for r in rows if mask[r] > 0), dtype=np.int64)
    return dict(hidden=hidden, weight=weight, targets=targets, mask=mask, grad=grad,
                dev=(hd, wd, yd, md, gd), logp=logp.cpu(), lse=lse.cpu(), dh=dh.cpu(), dw=dw,
                rows=rows, w64=oracle.bf16_bits_to_f64(weight))


def test_forward_and_dh_sampled_rows(big):
    rows, w64 = big["rows"], big["w64"]
    h64 = f64(big["hidden"][rows])
    y = big["targets"][rows].numpy()
    lp_o, lse_o = oracle.linear_logp_fwd_parallel(h64, w64, y, None, T)
    dl = np.abs(big["logp"].double().numpy()[rows] - lp_o)
    dz = np.abs(big["lse"].double().numpy()[rows] - lse_o)
    g32 = np.float32(big["grad"][rows]).astype(np.float64)
    dh_o = oracle.linear_logp_bwd_dh_parallel(h64, w64, y, None, g32, lse_o, T)
    e = rel_l2(big["dh"][rows], dh_o)
    print("N=65536: %d sampled rows, max |dlogp| %.3e, max |dlse| %.3e, dh rel-L2 %.3e"
          % (len(rows), dl.max(), dz.max(), e))
    assert dl.max() <= LOGP_ATOL and dz.max() <= LOGP_ATOL
    assert e <= GRAD_REL_L2
    inactive = big["mask"].numpy() == 0
    assert np.all(big["logp"].numpy()[inactive] == 0) and torch.all(big["dh"][inactive] == 0)


def test_dweight_identity_and_run_to_run(big):
    dw = big["dw"]
    col = dw.double().sum(dim=0)
    rms = dw.double().pow(2).sum(dim=0).sqrt()
    worst = float((col.abs() / rms).max())
    print("N=65536: max |dW column sum| / column norm %.3e" % worst)
    assert worst <= 8 * 2.0 ** -8
    hd, wd, yd, md, gd = big["dev"]
    _, lse = rlk.linear_logp_fwd(hd, wd, yd, md, T)
    _, dw2 = rlk.linear_logp_bwd(hd, wd, yd, md, gd, lse, T)
    assert torch.equal(dw2.view(torch.int16), dw.view(torch.int16))


def test_rows_match_a_small_batch_bitwise(big):
    hd, wd, yd, md, gd = big["dev"]
    for a in (0, 31000, N - 300):
        b = a + 300
        logp, lse = rlk.linear_logp_fwd(hd[a:b], wd, yd[a:b], md[a:b], T)
        dh, _ = rlk.linear_logp_bwd(hd[a:b], wd, yd[a:b], md[a:b], gd[a:b], lse, T)
        assert same_bits(logp.cpu(), big["logp"][a:b]) and same_bits(lse.cpu(), big["lse"][a:b])
        assert same_bits(dh.cpu(), big["dh"][a:b])
