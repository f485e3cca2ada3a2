"""The audit entry point that allocates nothing (rlk_dlogp_audit_noalloc).

Some callers cannot call cudaMalloc -- a rollout engine that reserved nearly
all device memory for its KV cache at start-up, or a framework hook that may
only use the tensors it is handed -- so this variant keeps its scratch in a
fixed array inside the library instead of a caller workspace.  Checked here
through the C ABI against rlk_dlogp_audit on two calls in a row (the second,
smaller call must not see the first call's leftovers in the shared scratch),
with the tolerances of the audit parity tests.  This file is collected last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import rl_post_linear_gb300 as rlk
import workloads as wl

pytestmark = pytest.mark.gpu


def _decode(raw):
    r = rlk.AuditResult.from_buffer_copy(bytes(raw.cpu().numpy().tobytes()))
    return {f: getattr(r, f) for f, _ in rlk.AuditResult._fields_}


def _same(a, b, new, old, mask):
    assert a["active_count"] == b["active_count"]
    assert a["argmax_index"] == b["argmax_index"]
    assert a["max_abs_dlogp"] == b["max_abs_dlogp"]
    assert a["error_flags"] == b["error_flags"]
    act = mask.cpu().numpy() > 0
    mean_abs = float(np.mean(np.abs(new.cpu().double().numpy() - old.cpu().double().numpy())[act]))
    assert abs(a["mean_dlogp"] - b["mean_dlogp"]) <= 1e-6 * mean_abs + 1e-12
    assert abs(a["approx_kl"] - b["approx_kl"]) <= 1e-6 * abs(b["approx_kl"]) + 1e-15


def test_noalloc_matches_workspace_audit_twice():
    lib = rlk.load()
    d = torch.device("cuda:0")
    stream = torch.cuda.current_stream().cuda_stream
    for n, seed in ((3_000_001, 7), (5_003, 8)):
        new, old, mask = (t.to(d) for t in wl.audit_inputs(n, seed))
        ref = rlk.dlogp_audit(new, old, mask)
        res = torch.empty(rlk.AUDIT_RESULT_BYTES, dtype=torch.uint8, device=d)
        st = lib.rlk_dlogp_audit_noalloc(new.data_ptr(), old.data_ptr(), mask.data_ptr(), n,
                                         res.data_ptr(), ctypes.c_void_p(stream))
        assert st == rlk.RLK_OK
        torch.cuda.synchronize()
        got = _decode(res)
        assert got["active_count"] == int(mask.sum())
        _same(got, ref, new, old, mask)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = rlk.load()
    st = lib.rlk_dlogp_audit_noalloc(None, None, None, rlk.RLK_AUDIT_NOALLOC_MAX_N + 1, None, None)
    assert st == rlk.RLK_ERR_UNSUPPORTED
    d = torch.device("cuda:0")
    res = torch.empty(rlk.AUDIT_RESULT_BYTES, dtype=torch.uint8, device=d)
    z = torch.zeros(0, device=d)
    rlk.rlk_dlogp_audit_noalloc(z, z, None, res)
    torch.cuda.synchronize()
    r = _decode(res)
    assert r["active_count"] == 0 and r["argmax_index"] == -1 and math.isnan(r["mean_dlogp"])
