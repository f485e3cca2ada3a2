"""Benchmark: one step = the whole hot path on one batch of synthetic input.

A step runs, on one stream, the fused linear log-prob forward, the GRPO
clipped-ratio loss fragment (per-token upstream gradient, token-mean over the
active tokens), the masked dlogp audit of the new logp against the
rollout-side old logp, and the chunked-recompute backward -- all in
librlk.so kernels.

Workload (default): the Qwen3-8B-shaped LM head, N = 8192 tokens packed from
8 sequences, H = 4096, V = 151936, T = 0.7, targets sampled from the softmax
of the logits, all tokens active; old logp = forward logp + N(0, 0.01^2)
noise, advantages ~ N(0, 1) per sequence, eps = 0.2.  Inputs are synthetic
and seeded; W (1.245 GB) is larger than L2, so no flush is needed between
steps.

Output: one JSON line (rank 0).  ``value`` is whole-job active tokens per
second with inputs resident in HBM; ``e2e`` is the same metric through the C
ABI with the per-step inputs copied from pinned host memory and the result
read back inside the timed region (step i+1's inputs are copied on a second
stream while step i computes, into the other of two device input sets).  ``--impl reference`` times the fp64 CPU
oracle on a bounded token sample of the same workload instead.

Multi-GPU (torchrun): every rank scores its own batch (seed + rank); there is
no collective on the data path, only a barrier and a max over ranks of the
timed region (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "fused linear-logp tokens/s and TFLOP/s (fwd, bwd) on 1 GB300; % of bf16 dense peak"
GRPO_EPS = 0.2


# ----------------------------------------------------------------------------- environment

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.mark = 0

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            # nvidia-smi takes a moment to start: wait for its first sample (bounded) so the
            # samples kept cover the timed region, not the tool's start-up
            t0 = time.time()
            while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
                time.sleep(0.01)
        except OSError:
            self.proc = None
        self.mark = len(self.lines)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        kept = self.lines[self.mark:] or self.lines
        for ln in kept:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


def needs_remeasure(summary, world, device):
    """True when this rank's (or, under torchrun, any rank's) timed region saw hw_slowdown,
    hw_thermal_slowdown or sw_thermal_slowdown, or a median SM clock below 70% of the maximum
    with no reason active."""
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    flag = 0.0
    if set(summary["reasons"]) & bad:
        flag = 1.0
    elif (summary["sm_mhz"] is not None and summary["sm_max_mhz"]
          and not summary["reasons"] and summary["sm_mhz"] < 0.7 * summary["sm_max_mhz"]):
        flag = 1.0
    t = torch.tensor([flag], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return bool(t.item() > 0)


def max_over_ranks(values, world, device):
    """Element-wise max of per-rank timings (the job is as slow as its slowest rank)."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def rank_seed(seed, rank):
    """Each rank scores its own batch: weak scaling with no data-path collective."""
    return seed + rank


# ----------------------------------------------------------------------------- workload

def make_batch(seed, n_tokens=wl.QWEN_N):
    w = wl.qwen_fwd(seed, n_tokens=n_tokens, sample=True)
    noise, adv = wl.grpo_bwd_extras(w.n, w.seq_lens, seed)
    return w, noise, adv


# ----------------------------------------------------------------------------- our arm

def run_ours(args, world, rank, local):
    import rl_post_linear_gb300 as rlk
    from rl_post_linear_gb300 import build as rlk_build
    if rank == 0:
        rlk_build.build()
    if world > 1:
        torch.distributed.barrier()
    rlk.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    w, noise, adv = make_batch(rank_seed(args.seed, rank), args.tokens)
    n, h, v, T = w.n, w.h, w.v, w.temperature
    n_act = w.n_active
    hid = w.hidden.to(dev)
    wt = w.weight.to(dev)
    y = w.targets.to(dev)
    mask = w.mask.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    logp = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev)
    dh = torch.empty_like(hid)
    dw = torch.empty_like(wt)
    ws_f = torch.empty(rlk.rlk_linear_logp_fwd_workspace_bytes(n, h, v), dtype=torch.uint8,
                       device=dev)
    ws_b = torch.empty(rlk.rlk_linear_logp_bwd_workspace_bytes(n, h, v), dtype=torch.uint8,
                       device=dev)
    ws_a = torch.empty(rlk.rlk_dlogp_audit_workspace_bytes(n), dtype=torch.uint8, device=dev)
    audit = torch.empty(rlk.AUDIT_RESULT_BYTES, dtype=torch.uint8, device=dev)

    # input preparation: the rollout-side old logp (forward logp + noise) and advantages
    rlk.rlk_linear_logp_fwd(hid, wt, y, mask, T, logp, lse, ws_f, err)
    torch.cuda.synchronize()
    old = (logp.double() + torch.from_numpy(noise).to(dev)).float()
    advd = torch.from_numpy(adv).float().to(dev)
    g = torch.empty(n, dtype=torch.float32, device=dev)
    ws_l = torch.empty(rlk.rlk_grpo_clip_loss_workspace_bytes(n), dtype=torch.uint8, device=dev)
    loss_res = torch.empty(rlk.GRPO_RESULT_BYTES, dtype=torch.uint8, device=dev)
    scale = 1.0 / n_act                         # token mean over the batch's active tokens
    n_chunks = -(-v // 32768)
    # forward: row compaction (3, the step passes a mask) + GEMM + merge; loss 2; audit 2;
    # backward: row compaction (3) and the zeroing of inactive dh rows (1), target sort (2),
    # then per vocab chunk the three GEMM roles and the sort of the chunk's dominant
    # non-target classes (2)
    launches_per_step = 5 + 2 + 2 + 4 + 2 + 5 * n_chunks

    def step(ev=None, ins=None):
        h_t, y_t, m_t, old_t, adv_t = ins if ins is not None else (hid, y, mask, old, advd)
        if ev is not None:
            ev[0].record(stream)
        rlk.rlk_linear_logp_fwd(h_t, wt, y_t, m_t, T, logp, lse, ws_f, err)
        if ev is not None:
            ev[1].record(stream)
        rlk.rlk_grpo_clip_loss(logp, old_t, adv_t, m_t, GRPO_EPS, GRPO_EPS, scale, g, loss_res,
                               ws_l)
        rlk.rlk_dlogp_audit(logp, old_t, m_t, audit, ws_a)
        if ev is not None:
            ev[2].record(stream)
        rlk.rlk_linear_logp_bwd(h_t, wt, y_t, m_t, g, lse, T, dh, dw, ws_b, err)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    def timed_region():
        evs_ = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
                for _ in range(args.steps)]
        start_, stop_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as sampler:
            torch.cuda.synchronize()
            start_.record(stream)
            for i in range(args.steps):
                step(evs_[i])
            stop_.record(stream)
            torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        return evs_, start_, stop_, sampler

    evs, start, stop, clocks = timed_region()
    # A timed region that saw a hardware or thermal slowdown, or SM clocks far below the
    # maximum with no reason given (a clock lock left by someone else), is measured once
    # more; every rank takes the same decision.
    remeasured = None
    if needs_remeasure(clocks.summary(), world, dev):
        remeasured = {"first_ms_per_step": start.elapsed_time(stop) / args.steps,
                      "first_clocks": clocks.summary()}
        evs, start, stop, clocks = timed_region()
    total_ms = start.elapsed_time(stop)
    fwd_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    aud_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))   # loss fragment + audit
    bwd_ms = float(np.mean([e[2].elapsed_time(e[3]) for e in evs]))
    if int(err.item()) != 0:
        raise RuntimeError("device error word %#x" % int(err.item()))

    # e2e: per-step inputs from pinned host memory through the C ABI, results read back
    h_host = w.hidden.pin_memory()
    y_host = w.targets.pin_memory()
    m_host = w.mask.pin_memory()
    old_host = old.cpu().pin_memory()
    adv_host = advd.cpu().pin_memory()
    logp_host = torch.empty(n, dtype=torch.float32).pin_memory()
    audit_host = torch.empty(rlk.AUDIT_RESULT_BYTES, dtype=torch.uint8).pin_memory()
    loss_host = torch.empty(rlk.GRPO_RESULT_BYTES, dtype=torch.uint8).pin_memory()
    # Two device input sets: step i+1's inputs are copied on a second stream while step i
    # computes (a trainer's prefetch); every copy still lies inside the timed region.
    sets = [(torch.empty_like(hid), torch.empty_like(y), torch.empty_like(mask),
             torch.empty_like(old), torch.empty_like(advd)) for _ in range(2)]
    hosts = (h_host, y_host, m_host, old_host, adv_host)
    copy_stream = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]

    def prefetch(i):
        b = i % 2
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(free[b])      # step i-2 is done with this set
            for dst, src in zip(sets[b], hosts):
                dst.copy_(src, non_blocking=True)
            ready[b].record(copy_stream)

    def e2e_run(k, begin=None):
        if begin is not None:
            copy_stream.wait_event(begin)
        prefetch(0)
        for i in range(k):
            if i + 1 < k:
                prefetch(i + 1)
            b = i % 2
            stream.wait_event(ready[b])
            step(None, sets[b])
            free[b].record(stream)
            logp_host.copy_(logp, non_blocking=True)
            audit_host.copy_(audit, non_blocking=True)
            loss_host.copy_(loss_res, non_blocking=True)

    e2e_run(max(1, args.warmup))
    torch.cuda.synchronize()
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    e2e_run(args.steps, e_start)
    e_stop.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e_start.elapsed_time(e_stop)
    h2d = (h_host.numel() * 2 + y_host.numel() * 8 + m_host.numel() + old_host.numel() * 4
           + adv_host.numel() * 4)
    d2h = logp_host.numel() * 4 + audit_host.numel() + loss_host.numel()

    total_ms, e2e_ms, fwd_ms, aud_ms, bwd_ms = max_over_ranks(
        [total_ms, e2e_ms, fwd_ms, aud_ms, bwd_ms], world, dev)
    if rank != 0:
        return None

    pk = peaks()
    ms_step = total_ms / args.steps
    tok = n_act * world
    fwd_tflops = 2.0 * n_act * h * v / (fwd_ms * 1e-3) / 1e12
    bwd_tflops = 4.0 * n_act * h * v / (bwd_ms * 1e-3) / 1e12
    peak = pk["bf16_tflops_sustained"]
    audit_gbs = n * 26 / (aud_ms * 1e-3) / 1e9
    # roofline: the forward GEMM is the largest single launch, and the only GEMM whose entry
    # point holds one GEMM launch (plus a 0.4% merge), so events around it time it directly;
    # the backward group (15 GEMM launches + the target sort) is reported beside it
    out = {
        "metric": METRIC,
        "value": tok / (ms_step * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; Qwen3-8B-shaped LM head, random-init weights)",
        "config": {"workload": w.name + " fwd+GRPO loss+audit+bwd", "n_tokens": n,
                   "n_active": n_act, "hidden": h, "vocab": v, "temperature": T,
                   "seq_lens": w.seq_lens, "parallelism": "dp%d (independent batches)" % world,
                   "l2": "inputs larger than L2 (W = %.3f GB), no flush" % (v * h * 2 / 1e9)},
        "fwd": {"ms": fwd_ms, "tflops": fwd_tflops, "frac_of_peak": fwd_tflops / peak,
                "flops": 2.0 * n_act * h * v},
        "bwd": {"ms": bwd_ms, "tflops": bwd_tflops, "frac_of_peak": bwd_tflops / peak,
                "flops": 4.0 * n_act * h * v,
                "executed_tflops": 6.0 * n * h * v / (bwd_ms * 1e-3) / 1e12},
        "loss_and_audit": {"ms": aud_ms, "gbs": audit_gbs, "frac_of_hbm": audit_gbs / pk["hbm_gbs"],
                           "bytes": "N x (4+4+4+1+4 loss, 4+4+1 audit)"},
        "roofline": {"bound": "tensor", "kernel": "gemm_persistent_kernel<FwdPolicy>",
                     "achieved": fwd_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": fwd_tflops / peak, "traffic": recorded_traffic("fwd_gemm", n, v, h),
                     "peak_source": "%s bf16 sustained (MEASURED_PEAKS.json)" % pk["source"]},
        "roofline_bwd": {"bound": "tensor", "kernel": "backward group (dS, dh, dW GEMMs + sort)",
                         "achieved": bwd_tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": bwd_tflops / peak, "flops": "4*N_a*H*V algorithmic",
                         "traffic": None},
        "e2e": {"value": tok / (e2e_ms / args.steps * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
    }
    if remeasured is not None:
        out["remeasured"] = remeasured
    out["audit_hbm"] = {str(na): measure_audit(rlk, dev, na, pk["hbm_gbs"])
                        for na in (9_400_614, 1 << 26)}
    if not args.no_next_rows:
        out["next_rows"] = measure_next_rows(rlk, dev, pk, args.warmup, args.steps,
                                             (hid, wt, y, mask, T, n_act, logp, g, dh, dw, ws_f,
                                              ws_b))
    if not args.no_second_shape:
        del hid, wt, dh, dw, ws_b
        torch.cuda.empty_cache()
        out["deepseek_fwd"], out["deepseek_bwd"] = measure_deepseek(rlk, dev, peak, args.warmup,
                                                                    args.steps)
    if not args.no_cpu_baseline and world == 1:
        out["cpu_baseline"] = cpu_baseline(w, noise, adv, args.cpu_tokens)
    return out


def _time_calls(fn, warmup, steps, stream):
    """Mean device time of one call of fn (CUDA events on the launching stream)."""
    for _ in range(max(3, warmup)):
        fn()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def measure_next_rows(rlk, dev, pk, warmup, steps, state):
    """The rows built after the hot path, each timed alone on the Qwen-shaped batch (or at
    N = 2^26 for the per-token fragments), against the roofline that bounds it:
    the vocab-sharded forward (TP = 4 emulated on one GPU: four block launches and the
    fixed-order merge, checked bitwise against the unsharded logp) and backward (four block
    backwards and the dh merge), the data-parallel backward of four emulated ranks (fp32 dW
    partials and their rank-order merge), the entropy forward and
    backward, logp from existing fp32 / bf16 logits [8192, 151936], the extended audit and
    the clipped-ratio loss fragment."""
    from rl_post_linear_gb300 import tp
    hid, wt, y, mask, T, n_act, logp_ref, g, dh, dw, ws_f, ws_b = state
    n, h = hid.shape
    v = wt.shape[0]
    stream = torch.cuda.current_stream()
    peak, hbm = pk["bf16_tflops_sustained"], pk["hbm_gbs"]
    fwd_flops, bwd_flops = 2.0 * n_act * h * v, 4.0 * n_act * h * v
    res = {}

    # NEXT-1: TP = 4 emulated
    shards = tp.vocab_shards(v, 4)
    total = rlk.rlk_linear_logp_num_partials(v)
    partials = torch.empty(total, n, 2, dtype=torch.float32, device=dev)
    tl = torch.zeros(n, dtype=torch.float32, device=dev)
    lp4, lse4 = torch.empty_like(logp_ref), torch.empty_like(logp_ref)

    def tp_fwd():
        for start, size in shards:
            if size == 0:
                continue
            c0 = start // tp.CHUNK
            cnt = rlk.rlk_linear_logp_num_partials(size)
            rlk.rlk_linear_logp_fwd_shard(hid, wt[start:start + size], y, mask, start, T,
                                          partials[c0:c0 + cnt], tl)
        rlk.rlk_linear_logp_merge(partials, total, tl, y, mask, v, T, lp4, lse4)

    ms = _time_calls(tp_fwd, warmup, steps, stream)
    rlk.rlk_linear_logp_fwd(hid, wt, y, mask, T, logp_ref, None, ws_f)
    torch.cuda.synchronize()
    res["tp4_emulated_fwd"] = {
        "ms": ms, "tflops": fwd_flops / (ms * 1e-3) / 1e12,
        "frac_of_peak": fwd_flops / (ms * 1e-3) / 1e12 / peak,
        "bitwise_equal_to_unsharded": bool(torch.equal(lp4.view(torch.int32),
                                                       logp_ref.view(torch.int32))),
        "launches": len(shards) + 1}
    del partials

    # NEXT-1 backward: TP = 4 emulated (each vocab block's fp32 dh partial and its rows of
    # dW, then the fixed-order dh merge); the dW rows are bitwise the unsharded ones
    lse_m = torch.empty_like(logp_ref)
    rlk.rlk_linear_logp_fwd(hid, wt, y, mask, T, logp_ref, lse_m, ws_f)
    dh_parts = torch.empty(len(shards), n, h, dtype=torch.float32, device=dev)
    dw4, dh4 = torch.empty_like(wt), torch.empty_like(hid)
    ws_s = torch.empty(max(256, max(rlk.rlk_linear_logp_bwd_workspace_bytes(n, h, size)
                                    for _, size in shards)), dtype=torch.uint8, device=dev)

    def tp_bwd():
        for r, (start, size) in enumerate(shards):
            rlk.rlk_linear_logp_bwd_shard(hid, wt[start:start + size], y, mask, g, lse_m, start,
                                          v, T, dh_parts[r], dw4[start:start + size], ws_s)
        rlk.rlk_linear_logp_dh_merge(dh_parts, dh4)

    ms = _time_calls(tp_bwd, warmup, steps, stream)
    rlk.rlk_linear_logp_bwd(hid, wt, y, mask, g, lse_m, T, dh, dw, ws_b)
    torch.cuda.synchronize()
    res["tp4_emulated_bwd"] = {
        "ms": ms, "tflops": bwd_flops / (ms * 1e-3) / 1e12,
        "frac_of_peak": bwd_flops / (ms * 1e-3) / 1e12 / peak,
        "dw_bitwise_equal_to_unsharded": bool(torch.equal(dw4.view(torch.int16),
                                                          dw.view(torch.int16))),
        "dh_rel_diff_to_unsharded": float((dh4.float() - dh.float()).norm()
                                          / dh.float().norm())}
    del dh_parts, dw4, dh4, ws_s

    # Section 8(e): data parallelism over tokens emulated as 4 ranks of N/4 tokens, each an
    # unrounded fp32 dW partial, then the rank-order merge (reads 4 V H fp32, writes V H bf16)
    splits = [0, n // 4, n // 2, 3 * n // 4, n]
    parts = torch.empty(4, v, h, dtype=torch.float32, device=dev)
    dh_d, dw_d = torch.empty_like(hid), torch.empty_like(wt)
    ws_d = torch.empty(max(rlk.rlk_linear_logp_bwd_workspace_bytes(splits[r + 1] - splits[r], h, v)
                           for r in range(4)), dtype=torch.uint8, device=dev)

    def dp_partials():
        for r in range(4):
            a, b = splits[r], splits[r + 1]
            rlk.rlk_linear_logp_bwd_dw_partial(hid[a:b], wt, y[a:b], mask[a:b], g[a:b],
                                               lse_m[a:b], T, dh_d[a:b], parts[r], ws_d)

    def dp_bwd():
        dp_partials()
        rlk.rlk_linear_logp_dw_merge(parts, dw_d)

    ms = _time_calls(dp_bwd, warmup, steps, stream)
    ms_m = _time_calls(lambda: rlk.rlk_linear_logp_dw_merge(parts, dw_d), warmup, steps, stream)
    merge_bytes = 4 * v * h * 4 + v * h * 2
    res["dp4_emulated_bwd"] = {
        "ms": ms, "tflops": bwd_flops / (ms * 1e-3) / 1e12,
        "frac_of_peak": bwd_flops / (ms * 1e-3) / 1e12 / peak,
        "merge_ms": ms_m, "merge_gbs": merge_bytes / (ms_m * 1e-3) / 1e9,
        "merge_frac_of_hbm": merge_bytes / (ms_m * 1e-3) / 1e9 / hbm,
        "dw_rel_diff_to_whole_batch": float((dw_d.float() - dw.float()).norm()
                                            / dw.float().norm()),
        "note": "4 emulated ranks of N/4 tokens; fp32 partials 4 V H (9.96 GB) merged in rank "
                "order, rounded once"}
    del parts, dh_d, dw_d, ws_d
    torch.cuda.empty_cache()

    # NEXT-3: entropy forward and backward
    ent = torch.empty_like(logp_ref)
    lse_e = torch.empty_like(logp_ref)
    ms_f = _time_calls(lambda: rlk.rlk_linear_logp_entropy_fwd(hid, wt, y, mask, T, lp4, lse_e,
                                                               ent, ws_f),
                       warmup, steps, stream)
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    g_ent = torch.randn(n, device=dev, generator=gen) / n
    ws_eb = torch.empty(rlk.rlk_linear_logp_entropy_bwd_workspace_bytes(n, h, v),
                        dtype=torch.uint8, device=dev)
    ms_b = _time_calls(lambda: rlk.rlk_linear_logp_entropy_bwd(hid, wt, y, mask, g, g_ent, lse_e,
                                                               ent, T, dh, dw, ws_eb),
                       warmup, steps, stream)
    del ws_eb
    res["entropy_fwd"] = {"ms": ms_f, "tflops": fwd_flops / (ms_f * 1e-3) / 1e12,
                          "frac_of_peak": fwd_flops / (ms_f * 1e-3) / 1e12 / peak}
    # executed: the dS recompute (2 N H V) and the dh and dW GEMMs over the hi and lo planes
    # of dS (4 N H V each)
    ent_exec = 2.5 * bwd_flops
    res["entropy_bwd"] = {"ms": ms_b, "tflops": bwd_flops / (ms_b * 1e-3) / 1e12,
                          "frac_of_peak": bwd_flops / (ms_b * 1e-3) / 1e12 / peak,
                          "executed_tflops": ent_exec / (ms_b * 1e-3) / 1e12,
                          "executed_frac_of_peak": ent_exec / (ms_b * 1e-3) / 1e12 / peak}

    # NEXT-3: full-vocabulary KL against a reference head of the same shape (a frozen
    # reference policy); forward 2 N V (H + Hr) FLOP, backward 4 N H V algorithmic (dh, dW;
    # the recompute of both heads, 2 N V (H + Hr), is executed on top)
    hid_r = (hid.float() + torch.randn(hid.shape, device=dev, generator=gen)
             * 0.1).to(torch.bfloat16)
    wt_r = (wt.float() + torch.randn(wt.shape, device=dev, generator=gen)
            * 0.005).to(torch.bfloat16)
    kl, kl_r, lse_p, lse_q = (torch.empty_like(logp_ref) for _ in range(4))
    ws_kl = torch.empty(rlk.rlk_linear_kl_fwd_workspace_bytes(n, v), dtype=torch.uint8,
                        device=dev)
    ms_f = _time_calls(lambda: rlk.rlk_linear_kl_fwd(hid, wt, hid_r, wt_r, None, mask, T, T, kl,
                                                     kl_r, lse_p, lse_q, None, ws_kl),
                       warmup, steps, stream)
    g_kl = torch.randn(n, device=dev, generator=gen) / n
    del ws_kl
    ws_klb = torch.empty(rlk.rlk_linear_kl_bwd_workspace_bytes(n, h, v), dtype=torch.uint8,
                         device=dev)
    ms_b = _time_calls(lambda: rlk.rlk_linear_kl_bwd(hid, wt, hid_r, wt_r, mask, g_kl, g_kl,
                                                     lse_p, lse_q, kl, T, T, dh, dw, ws_klb),
                       warmup, steps, stream)
    kl_fwd_flops = 2.0 * n_act * v * (h + h)
    res["kl_fwd"] = {"ms": ms_f, "tflops": kl_fwd_flops / (ms_f * 1e-3) / 1e12,
                     "frac_of_peak": kl_fwd_flops / (ms_f * 1e-3) / 1e12 / peak,
                     "reference_head": "same shape as the policy head",
                     "mean_kl": float(kl.float().mean())}
    # executed: both heads recomputed (2 N V (H + Hr)) and the dh and dW GEMMs over the hi
    # and lo planes of dS (4 N H V each)
    kl_exec = 2.0 * bwd_flops + kl_fwd_flops
    res["kl_bwd"] = {"ms": ms_b, "tflops": bwd_flops / (ms_b * 1e-3) / 1e12,
                     "frac_of_peak": bwd_flops / (ms_b * 1e-3) / 1e12 / peak,
                     "executed_tflops": kl_exec / (ms_b * 1e-3) / 1e12,
                     "executed_frac_of_peak": kl_exec / (ms_b * 1e-3) / 1e12 / peak}
    del hid_r, wt_r, ws_klb
    torch.cuda.empty_cache()

    # NEXT-4: logp from existing logits, dense rows; bytes = the logits + targets, mask, out
    for name, dt, es in (("logits_fp32", torch.float32, 4), ("logits_bf16", torch.bfloat16, 2)):
        logits = (torch.randn(n, v, device=dev, generator=gen) * 2.0).to(dt)
        nbytes = n * v * es + n * (8 + 1 + 4 + 4)
        ms = _time_calls(lambda: rlk.rlk_logp_from_logits(logits, None, y, mask, T, lp4, lse4),
                         warmup, steps, stream)
        res["logp_from_" + name] = {"ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9,
                                    "frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm,
                                    "bytes": nbytes, "shape": [n, v]}
        del logits
    torch.cuda.empty_cache()

    # NEXT-4 extended audit and NEXT-2 loss fragment at N = 2^26 (inputs larger than L2)
    na = 1 << 26
    new, old, m = (t.to(dev) for t in wl.audit_inputs(na, 0))
    r_ext = torch.empty(rlk.AUDIT_EXT_RESULT_BYTES, dtype=torch.uint8, device=dev)
    ws_e = torch.empty(rlk.rlk_dlogp_audit_ext_workspace_bytes(na), dtype=torch.uint8,
                       device=dev)
    ms = _time_calls(lambda: rlk.rlk_dlogp_audit_ext(new, old, m, None, GRPO_EPS, r_ext, ws_e),
                     warmup, steps, stream)
    res["audit_ext_2p26"] = {"ms": ms, "gbs": na * 9 / (ms * 1e-3) / 1e9,
                             "frac_of_hbm": na * 9 / (ms * 1e-3) / 1e9 / hbm,
                             "bytes": na * 9,
                             "note": "algorithmic 9 B/token: the inputs are read once by the "
                                     "main pass (plus a sample of 128 slices); the keys inside "
                                     "the percentiles' windows (a few % of the tokens) are "
                                     "listed and radix-selected"}
    adv = torch.randn(na, device=dev, generator=gen)
    grad = torch.empty(na, dtype=torch.float32, device=dev)
    r_loss = torch.empty(rlk.GRPO_RESULT_BYTES, dtype=torch.uint8, device=dev)
    ws_l = torch.empty(rlk.rlk_grpo_clip_loss_workspace_bytes(na), dtype=torch.uint8, device=dev)
    ms = _time_calls(lambda: rlk.rlk_grpo_clip_loss(new, old, adv, m, GRPO_EPS, GRPO_EPS,
                                                    1.0 / na, grad, r_loss, ws_l),
                     warmup, steps, stream)
    res["grpo_loss_2p26"] = {"ms": ms, "gbs": na * 17 / (ms * 1e-3) / 1e9,
                             "frac_of_hbm": na * 17 / (ms * 1e-3) / 1e9 / hbm,
                             "bytes": na * 17, "note": "13 B read + 4 B gradient written per token"}
    return res


def measure_deepseek(rlk, dev, peak, warmup, steps):
    """The second workload of the pages' shapes: the DeepSeek-style LM head forward and
    backward (N = 16384, H = 7168, V = 129280, 20% of tokens masked, T = 1); W (1.85 GB)
    exceeds L2.  TFLOP/s counts the active tokens' work, 2 N_a H V forward and 4 N_a H V
    backward (upstream gradient N(0, 1) / N_a on the active tokens)."""
    w = wl.deepseek_fwd(0)
    hid, wt = w.hidden.to(dev), w.weight.to(dev)
    y, mask = w.targets.to(dev), w.mask.to(dev)
    logp = torch.empty(w.n, dtype=torch.float32, device=dev)
    lse = torch.empty_like(logp)
    ws = torch.empty(rlk.rlk_linear_logp_fwd_workspace_bytes(w.n, w.h, w.v), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        rlk.rlk_linear_logp_fwd(hid, wt, y, mask, w.temperature, logp, lse, ws)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        rlk.rlk_linear_logp_fwd(hid, wt, y, mask, w.temperature, logp, lse, ws)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    act = 2.0 * w.n_active * w.h * w.v / (ms * 1e-3) / 1e12
    fwd = {"workload": w.name, "n_active": w.n_active, "ms": ms,
           "tokens_per_s": w.n_active / (ms * 1e-3), "tflops_active": act,
           "frac_of_peak_active": act / peak,
           "note": "masked rows are compacted away before the GEMM (ceil(N_a/256) row tiles)"}

    g_host = np.random.default_rng(5).standard_normal(w.n).astype(np.float32) / w.n_active
    g_host[w.mask.numpy() == 0] = 0.0
    g = torch.from_numpy(g_host).to(dev)
    dh, dw = torch.empty_like(hid), torch.empty_like(wt)
    del ws
    ws_b = torch.empty(rlk.rlk_linear_logp_bwd_workspace_bytes(w.n, w.h, w.v), dtype=torch.uint8,
                       device=dev)
    for _ in range(warmup):
        rlk.rlk_linear_logp_bwd(hid, wt, y, mask, g, lse, w.temperature, dh, dw, ws_b)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        rlk.rlk_linear_logp_bwd(hid, wt, y, mask, g, lse, w.temperature, dh, dw, ws_b)
    b.record(stream)
    torch.cuda.synchronize()
    ms_b = a.elapsed_time(b) / steps
    act_b = 4.0 * w.n_active * w.h * w.v / (ms_b * 1e-3) / 1e12
    bwd = {"workload": w.name.replace("fwd", "bwd"), "n_active": w.n_active, "ms": ms_b,
           "tokens_per_s": w.n_active / (ms_b * 1e-3), "tflops_active": act_b,
           "frac_of_peak_active": act_b / peak,
           "note": "masked rows are compacted away before the three GEMMs of each chunk"}
    return fwd, bwd


def measure_audit(rlk, dev, n, hbm_gbs, reps=20):
    """The audit alone at N tokens: 9 algorithmic bytes per token (new, old, mask); the
    median of `reps` calls, each timed alone (the mean is reported beside it).  L2 is
    flushed before every timed launch pair (outside the events): a 2 GB write, then a 2 GB
    read that evicts the dirty lines, so that no write-back lands inside the timed region
    and inputs that fit in L2 are read from DRAM.  (After a 256 MB write and read some
    dirty lines stayed in L2: the audit at 2^26 then measured 104.5 against 96.3 us.)
    The flush also keeps the GPU busy while the host enqueues the audit (about 14 us of
    host time a call), so the events do not time the host's launch latency."""
    new, old, mask = (t.to(dev) for t in wl.audit_inputs(n, 0))
    res = torch.empty(rlk.AUDIT_RESULT_BYTES, dtype=torch.uint8, device=dev)
    ws = torch.empty(rlk.rlk_dlogp_audit_workspace_bytes(n), dtype=torch.uint8, device=dev)
    flush = torch.empty(2048 << 20, dtype=torch.uint8, device=dev)
    sweep = torch.empty(512 << 20, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        rlk.rlk_dlogp_audit(new, old, mask, res, ws)
    ms = []
    for _ in range(reps):
        flush.zero_()
        sweep.sum()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        rlk.rlk_dlogp_audit(new, old, mask, res, ws)
        b.record(stream)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    t = float(np.median(ms))
    gbs = n * 9 / (t * 1e-3) / 1e9
    return {"ms": t, "ms_mean": float(np.mean(ms)), "reps": reps, "gbs": gbs,
            "frac_of_hbm": gbs / hbm_gbs, "bytes": n * 9,
            "l2": "flushed (2 GB write + 2 GB read) before each launch pair"}


def measure_audit_ext(rlk, dev, n, hbm_gbs, warmup=3, steps=10):
    """The extended audit (exact percentiles, ratio0, clipfrac0) alone at N tokens, inputs
    resident, calls back to back."""
    new, old, m = (t.to(dev) for t in wl.audit_inputs(n, 0))
    r_ext = torch.empty(rlk.AUDIT_EXT_RESULT_BYTES, dtype=torch.uint8, device=dev)
    ws_e = torch.empty(rlk.rlk_dlogp_audit_ext_workspace_bytes(n), dtype=torch.uint8, device=dev)
    ms = _time_calls(lambda: rlk.rlk_dlogp_audit_ext(new, old, m, None, GRPO_EPS, r_ext, ws_e),
                     warmup, steps, torch.cuda.current_stream())
    gbs = n * 9 / (ms * 1e-3) / 1e9
    return {"ms": ms, "gbs": gbs, "frac_of_hbm": gbs / hbm_gbs, "bytes": n * 9}


def run_audit_only():
    """The audit rows of the workload table alone (for profiling the audit kernels): the
    base audit, then the extended audit, at N = 9,400,614 and 2^26."""
    import rl_post_linear_gb300 as rlk
    from rl_post_linear_gb300 import build as rlk_build
    rlk_build.build()
    rlk.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pk = peaks()
    sizes = (9_400_614, 1 << 26)
    out = {"audit_hbm": {str(na): measure_audit(rlk, dev, na, pk["hbm_gbs"]) for na in sizes}}
    out["audit_ext"] = {str(na): measure_audit_ext(rlk, dev, na, pk["hbm_gbs"]) for na in sizes}
    return out


def recorded_traffic(kernel, n, v, h):
    """DRAM bytes per launch of `kernel` at this (N, V, H), from the committed ncu summary
    (profiles/traffic.txt: kernel N V H bytes source-hash), or None if the kernel source has
    changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    cur = source_hash(kernel)
    for line in open(path):
        parts = line.split()
        if (len(parts) == 6 and parts[0] == kernel and parts[1:4] == [str(n), str(v), str(h)]
                and parts[5] == cur):
            return float(parts[4])
    return None


KERNEL_SOURCES = {"fwd_gemm": ("fwd.cu", "gemm.cuh", "ptx.cuh", "rlk_internal.h")}


def source_hash(kernel="fwd_gemm"):
    """Hash of the source files that define `kernel` (a changed kernel voids old counters)."""
    d = os.path.join(ROOT, "rl_post_linear_gb300", "csrc")
    hsh = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        hsh.update(open(os.path.join(d, f), "rb").read())
    return hsh.hexdigest()[:16]


# ----------------------------------------------------------------------------- CPU oracle legs

def oracle_step_sample(w, noise, adv, tokens, threads):
    """One oracle step (fwd, GRPO loss, audit, bwd with all V rows of dW) over the first
    `tokens` tokens of the batch, timed.  Everything it consumes is the oracle's own: the
    rollout-side old logp is its forward logp plus the workload's noise, formed before the
    timed region from an untimed oracle forward."""
    import oracle
    h64 = oracle.bf16_bits_to_f64(w.hidden[:tokens])
    w64 = getattr(w, "_w64", None)
    if w64 is None:
        w64 = oracle.bf16_bits_to_f64(w.weight)
        w._w64 = w64
    y = w.targets[:tokens].numpy()
    m = w.mask[:tokens].numpy()
    old = getattr(w, "_old_sample", None)
    if old is None or len(old) != tokens:
        lp0, _ = oracle.linear_logp_fwd_parallel(h64, w64, y, m, w.temperature, threads)
        old = (lp0 + noise[:tokens]).astype(np.float32).astype(np.float64)
        w._old_sample = old
    n_act = max(int(m.sum()), 1)
    t0 = time.perf_counter()
    lp, lse = oracle.linear_logp_fwd_parallel(h64, w64, y, m, w.temperature, threads)
    gg, _ = oracle.grpo_clip(lp, old, adv[:tokens], m, GRPO_EPS, GRPO_EPS, 1.0 / n_act)
    oracle.dlogp_audit(lp.astype(np.float32), old.astype(np.float32), m)
    oracle.linear_logp_bwd_dh_parallel(h64, w64, y, m, gg, lse, w.temperature, threads)
    oracle.linear_logp_bwd_dw_blocks(h64, w64, y, m, gg, lse, w.temperature, 0, w.v,
                                     lambda v0, blk: None, threads=threads)
    return time.perf_counter() - t0


def cpu_cores():
    return max(1, len(os.sched_getaffinity(0)))


def cpu_baseline(w, noise, adv, tokens):
    cores = cpu_cores()
    tokens = tokens or cores
    secs = oracle_step_sample(w, noise, adv, tokens, cores)
    return {"value": tokens / secs, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "first %d tokens of the batch, one full oracle step (fwd, GRPO loss, "
                      "audit, bwd with all %d dW rows), fp64, %.1f s" % (tokens, w.v, secs)}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    w, noise, adv = make_batch(args.seed, args.tokens)
    tokens = args.cpu_tokens or cpu_cores()
    oracle_step_sample(w, noise, adv, tokens, cpu_cores())      # warm-up: W conversion, old logp
    for _ in range(args.warmup - 1):
        oracle_step_sample(w, noise, adv, tokens, cpu_cores())
    times = [oracle_step_sample(w, noise, adv, tokens, cpu_cores()) for _ in range(args.steps)]
    secs = float(np.mean(times))
    val = tokens / secs
    return {
        "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; Qwen3-8B-shaped LM head, random-init weights)",
        "impl": "reference",
        "config": {"workload": w.name + " fwd+GRPO loss+audit+bwd", "n_tokens": w.n,
                   "n_active": w.n_active, "hidden": w.h, "vocab": w.v,
                   "temperature": w.temperature},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cpu_cores(),
                         "kind": "oracle",
                         "sample": "first %d tokens per step, full oracle step (fwd, GRPO loss, "
                                   "audit, bwd with all %d dW rows)" % (tokens, w.v)},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--tokens", type=int, default=wl.QWEN_N)
    ap.add_argument("--cpu-tokens", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-second-shape", action="store_true",
                    help="leave out the DeepSeek-shaped forward measurement")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="leave out the TP-emulated, entropy, logits, extended-audit and loss "
                         "measurements")
    ap.add_argument("--audit-only", action="store_true",
                    help="time only the masked audit at N = 9,400,614 and 2^26 (one GPU)")
    args = ap.parse_args()
    if args.audit_only:
        print(json.dumps(run_audit_only()))
        return
    world, rank, local = dist_env()
    if world > 1 and args.impl == "ours":
        torch.distributed.init_process_group("nccl")
    try:
        out = run_reference(args, world, rank) if args.impl == "reference" else \
            run_ours(args, world, rank, local)
        if out is not None:
            print(json.dumps(out))
    finally:
        if world > 1 and args.impl == "ours":
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
