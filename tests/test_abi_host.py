"""Host-side checks of the C ABI that need no GPU.

The library must build for sm_103a, load, export every function that
include/rlk.h declares, answer workspace queries, and reject invalid
arguments synchronously -- before it touches the CUDA runtime -- with the
documented status codes (explicit failure, no fallback: "RL-Kernel
integration roadmap for vime", linear_logp consistency target).
"""
import ctypes

import pytest

import rl_post_linear_gb300 as rlk
from rl_post_linear_gb300 import build as rlk_build


@pytest.fixture(scope="module")
def lib():
    rlk_build.build()
    return rlk.load()


def test_exports_every_declared_symbol(lib):
    names = rlk.declared_functions()
    assert set(names) >= {"rlk_linear_logp_fwd", "rlk_linear_logp_bwd", "rlk_dlogp_audit",
                          "rlk_linear_logp_fwd_workspace_bytes",
                          "rlk_linear_logp_bwd_workspace_bytes",
                          "rlk_dlogp_audit_workspace_bytes", "rlk_contract_string",
                          "rlk_status_string"}
    for n in names:
        assert hasattr(lib, n), n


def test_contract_and_status_strings(lib):
    s = rlk.rlk_contract_string()
    assert "sm_103a" in s and "no split-K" in s and "no float atomics" in s
    assert rlk.status_string(rlk.RLK_OK) == "RLK_OK"
    assert rlk.status_string(rlk.RLK_ERR_WORKSPACE) == "RLK_ERR_WORKSPACE"
    assert ctypes.sizeof(rlk.AuditResult) == 40


def test_workspace_queries(lib):
    # forward: 1024-column vocab chunks, (max, sum) float2 and the entropy sum per chunk and
    # row, plus a target logit; then the compaction of a masked batch: two int32 row lists,
    # per-1024-row block counts, the active count and the compacted bf16 copy of h
    n, v, h = 8192, 151936, 4096
    up = lambda x: -(-x // 256) * 256
    chunks = -(-(-(-v // 256)) // 4)
    expect = (up(chunks * n * 8) + up(chunks * n * 4) + up(n * 4) + 2 * up(n * 4)
              + up(-(-n // 1024) * 4) + up(4) + up(n * h * 2))
    assert rlk.rlk_linear_logp_fwd_workspace_bytes(n, h, v) == expect
    # backward: dS chunk [N, 32768] bf16 + fp32 dh accumulator + two int32 lists
    assert rlk.rlk_linear_logp_bwd_workspace_bytes(n, 4096, v) >= n * 32768 * 2 + n * 4096 * 4
    assert rlk.rlk_dlogp_audit_workspace_bytes(0) >= 256
    assert rlk.rlk_dlogp_audit_workspace_bytes(9400614) >= 2296 * 40
    assert rlk.rlk_linear_logp_fwd_workspace_bytes(-1, 64, 10) == 0


FAKE = 1 << 20          # a 16-byte aligned non-null address; validation never dereferences


def _fwd(lib, **kw):
    a = dict(hidden=FAKE, weight=FAKE, targets=FAKE, mask=None, N=4, H=64, V=10, T=1.0, logp=FAKE,
             lse=None, ws=FAKE, ws_bytes=1 << 20, err=None, stream=None)
    a.update(kw)
    return lib.rlk_linear_logp_fwd(a["hidden"], a["weight"], a["targets"], a["mask"], a["N"],
                                   a["H"], a["V"], a["T"], a["logp"], a["lse"], a["ws"],
                                   a["ws_bytes"], a["err"], a["stream"])


def test_forward_argument_errors(lib):
    assert _fwd(lib, H=100) == rlk.RLK_ERR_UNSUPPORTED
    assert _fwd(lib, H=0) == rlk.RLK_ERR_INVALID_VALUE
    assert _fwd(lib, T=0.0) == rlk.RLK_ERR_INVALID_VALUE
    assert _fwd(lib, T=-1.0) == rlk.RLK_ERR_INVALID_VALUE
    assert _fwd(lib, T=float("nan")) == rlk.RLK_ERR_INVALID_VALUE
    assert _fwd(lib, T=float("inf")) == rlk.RLK_ERR_INVALID_VALUE
    assert _fwd(lib, V=0) == rlk.RLK_ERR_INVALID_VALUE
    assert _fwd(lib, N=-1) == rlk.RLK_ERR_INVALID_VALUE
    assert _fwd(lib, N=1 << 31) == rlk.RLK_ERR_INVALID_VALUE
    assert _fwd(lib, N=(1 << 31) - (1 << 16) + 1) == rlk.RLK_ERR_INVALID_VALUE
    assert _fwd(lib, V=(1 << 31) - (1 << 16) + 1) == rlk.RLK_ERR_INVALID_VALUE
    assert _fwd(lib, hidden=None) == rlk.RLK_ERR_INVALID_VALUE
    assert _fwd(lib, targets=None) == rlk.RLK_ERR_INVALID_VALUE
    assert _fwd(lib, logp=None) == rlk.RLK_ERR_INVALID_VALUE
    assert _fwd(lib, hidden=FAKE + 2) == rlk.RLK_ERR_INVALID_VALUE
    assert _fwd(lib, weight=FAKE + 8) == rlk.RLK_ERR_INVALID_VALUE
    assert _fwd(lib, ws=None) == rlk.RLK_ERR_WORKSPACE
    assert _fwd(lib, ws=FAKE + 16) == rlk.RLK_ERR_WORKSPACE
    assert _fwd(lib, ws_bytes=16) == rlk.RLK_ERR_WORKSPACE
    # N = 0 is a valid no-op even with NULL buffers
    assert _fwd(lib, N=0, hidden=None, targets=None, logp=None, ws=None) == rlk.RLK_OK


def test_backward_and_audit_argument_errors(lib):
    def bwd(**kw):
        a = dict(hidden=FAKE, weight=FAKE, targets=FAKE, mask=None, g=FAKE, lse=FAKE, N=4, H=64,
                 V=10, T=0.7, dh=FAKE, dw=FAKE, ws=FAKE, ws_bytes=1 << 30, err=None, stream=None)
        a.update(kw)
        return lib.rlk_linear_logp_bwd(a["hidden"], a["weight"], a["targets"], a["mask"], a["g"],
                                       a["lse"], a["N"], a["H"], a["V"], a["T"], a["dh"], a["dw"],
                                       a["ws"], a["ws_bytes"], a["err"], a["stream"])

    assert bwd(H=96) == rlk.RLK_ERR_UNSUPPORTED
    assert bwd(g=None) == rlk.RLK_ERR_INVALID_VALUE
    assert bwd(lse=None) == rlk.RLK_ERR_INVALID_VALUE
    assert bwd(dh=FAKE + 4) == rlk.RLK_ERR_INVALID_VALUE
    assert bwd(dw=None) == rlk.RLK_ERR_INVALID_VALUE
    assert bwd(ws_bytes=1000) == rlk.RLK_ERR_WORKSPACE
    assert bwd(N=0, hidden=None) == rlk.RLK_OK
    assert lib.rlk_dlogp_audit(FAKE, FAKE, None, -1, FAKE, FAKE, 1 << 20, None) == \
        rlk.RLK_ERR_INVALID_VALUE
    assert lib.rlk_dlogp_audit(FAKE, FAKE, None, 10, None, FAKE, 1 << 20, None) == \
        rlk.RLK_ERR_INVALID_VALUE
    assert lib.rlk_dlogp_audit(None, FAKE, None, 10, FAKE, FAKE, 1 << 20, None) == \
        rlk.RLK_ERR_INVALID_VALUE
    assert lib.rlk_dlogp_audit(FAKE, FAKE, None, 10, FAKE, FAKE, 8, None) == rlk.RLK_ERR_WORKSPACE
    # the extended audit counts its selection in 32 bits: N below 2^32
    ext = lib.rlk_dlogp_audit_ext
    assert ext(FAKE, FAKE, None, 1 << 32, None, 0, 0.2, FAKE, FAKE, 1 << 40, None) == \
        rlk.RLK_ERR_UNSUPPORTED
    assert ext(FAKE, FAKE, None, -1, None, 0, 0.2, FAKE, FAKE, 1 << 40, None) == \
        rlk.RLK_ERR_INVALID_VALUE
    assert ext(FAKE, FAKE, None, 10, None, 0, -0.1, FAKE, FAKE, 1 << 40, None) == \
        rlk.RLK_ERR_INVALID_VALUE
    assert ext(FAKE, FAKE, None, 10, None, 0, 0.2, FAKE, FAKE, 8, None) == rlk.RLK_ERR_WORKSPACE


def test_binding_refuses_cpu_tensors(lib):
    import torch
    h = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        rlk.linear_logp_fwd(h, torch.zeros(10, 64, dtype=torch.bfloat16),
                            torch.zeros(4, dtype=torch.int64))
