"""One training step -- forward, clipped-ratio loss fragment, audit, backward -- captured
in a CUDA graph and replayed.

Every entry point only enqueues work on the caller's stream, on caller-owned buffers,
and never waits on the host (a masked batch's active-row count stays on the device), so
a trainer can capture the step once and replay it.  The replay must give, bit for bit,
what the eager calls give, and must read the inputs' current contents at each replay.
"""
import numpy as np
import pytest
import torch

import rl_post_linear_gb300 as rlk
import workloads as wl
from helpers import dev, same_bits

pytestmark = pytest.mark.gpu

N, H, V, T, EPS = 700, 256, 40000, 0.8, 0.2


def _buffers(seed):
    d = dev()
    hid = wl.normal_bf16((N, H), seed, wl.S_HIDDEN).to(d)
    wt = wl.normal_bf16((V, H), seed, wl.S_WEIGHT, std=0.05).to(d)
    y = wl.uniform_targets(N, V, seed).to(d)
    rng = np.random.default_rng(seed)
    mask = torch.from_numpy((rng.random(N) < 0.8).astype(np.uint8)).to(d)
    old = torch.from_numpy(rng.normal(-8.0, 1.0, N).astype(np.float32)).to(d)
    adv = torch.from_numpy(rng.normal(0.0, 1.0, N).astype(np.float32)).to(d)
    b = {
        "hid": hid, "wt": wt, "y": y, "mask": mask, "old": old, "adv": adv,
        "logp": torch.empty(N, dtype=torch.float32, device=d),
        "lse": torch.empty(N, dtype=torch.float32, device=d),
        "g": torch.empty(N, dtype=torch.float32, device=d),
        "dh": torch.empty_like(hid), "dw": torch.empty_like(wt),
        "loss": torch.empty(rlk.GRPO_RESULT_BYTES, dtype=torch.uint8, device=d),
        "audit": torch.empty(rlk.AUDIT_RESULT_BYTES, dtype=torch.uint8, device=d),
        "err": torch.zeros(1, dtype=torch.int32, device=d),
        "ws_f": torch.empty(rlk.rlk_linear_logp_fwd_workspace_bytes(N, H, V), dtype=torch.uint8,
                            device=d),
        "ws_b": torch.empty(rlk.rlk_linear_logp_bwd_workspace_bytes(N, H, V), dtype=torch.uint8,
                            device=d),
        "ws_a": torch.empty(rlk.rlk_dlogp_audit_workspace_bytes(N), dtype=torch.uint8, device=d),
        "ws_l": torch.empty(rlk.rlk_grpo_clip_loss_workspace_bytes(N), dtype=torch.uint8,
                            device=d),
    }
    return b


def _step(b):
    rlk.rlk_linear_logp_fwd(b["hid"], b["wt"], b["y"], b["mask"], T, b["logp"], b["lse"],
                            b["ws_f"], b["err"])
    n_act = 1.0 / max(1, N)
    rlk.rlk_grpo_clip_loss(b["logp"], b["old"], b["adv"], b["mask"], EPS, EPS, n_act, b["g"],
                           b["loss"], b["ws_l"])
    rlk.rlk_dlogp_audit(b["logp"], b["old"], b["mask"], b["audit"], b["ws_a"])
    rlk.rlk_linear_logp_bwd(b["hid"], b["wt"], b["y"], b["mask"], b["g"], b["lse"], T, b["dh"],
                            b["dw"], b["ws_b"], b["err"])


OUTS = ("logp", "lse", "g", "dh", "dw", "loss", "audit")


def _snapshot(b):
    torch.cuda.synchronize()
    return {k: b[k].clone() for k in OUTS}


def _poison(b):
    for k in OUTS:
        b[k].view(torch.uint8).fill_(0xFF)


def test_step_graph_replay_matches_eager():
    b = _buffers(81)
    _step(b)
    eager = _snapshot(b)
    assert int(b["err"].item()) == 0
    # warm up on a side stream, then capture (the usual order for torch's capture)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _step(b)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _step(b)
    _poison(b)
    graph.replay()
    replayed = _snapshot(b)
    for k in OUTS:
        assert same_bits(replayed[k].cpu(), eager[k].cpu()), k
    # new tokens (hidden rows, targets, mask, old logp, advantages) copied into the same
    # buffers: the replay reads them; the eager reference runs on its own buffers with the
    # same contents (and the same head)
    ref = _buffers(82)
    ref["wt"].copy_(b["wt"])
    for k in ("hid", "y", "mask", "old", "adv"):
        b[k].copy_(ref[k])
    _step(ref)
    eager_ref = _snapshot(ref)
    _poison(b)
    graph.replay()
    replayed2 = _snapshot(b)
    assert int(b["err"].item()) == 0
    for k in OUTS:
        assert same_bits(replayed2[k].cpu(), eager_ref[k].cpu()), k
    assert not same_bits(replayed2["logp"].cpu(), replayed["logp"].cpu())
