"""GB300-native fused linear selected-token log-prob (sm_103a).

A thin ctypes binding over ``librlk.so``, whose C ABI is ``include/rlk.h``.
Each ``rlk_*`` function here has the name and argument order of the C entry
point and only marshals torch tensors into pointers, sizes and the current
CUDA stream; all arithmetic runs in the library's kernels.  There is no CPU
path: if the library is missing or the device is not an sm_103 GPU, the calls
raise.

``linear_logp`` wraps forward and backward in a ``torch.autograd.Function``
for training code ("RL-Kernel integration roadmap for vime", linear_logp: a
forward-plus-backward training operator whose forward returns the selected
logp and keeps what the backward needs -- here the per-row lse).
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librlk.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "rlk.h")

RLK_OK, RLK_ERR_INVALID_VALUE, RLK_ERR_UNSUPPORTED, RLK_ERR_WORKSPACE, RLK_ERR_LAUNCH = range(5)
RLK_DEVERR_TARGET_RANGE = 0x1
RLK_DEVERR_WAIT_TIMEOUT = 0x2
RLK_AUDIT_NOALLOC_MAX_N = 1 << 27

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_lib = None


class RlkError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s" % (fn, status_string(status)))


class AuditResult(ctypes.Structure):
    """Mirror of rlk_audit_result_t."""
    _fields_ = [
        ("active_count", ctypes.c_int64),
        ("argmax_index", ctypes.c_int64),
        ("mean_dlogp", ctypes.c_double),
        ("approx_kl", ctypes.c_double),
        ("max_abs_dlogp", ctypes.c_float),
        ("error_flags", ctypes.c_uint32),
    ]


AUDIT_RESULT_BYTES = ctypes.sizeof(AuditResult)


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load librlk.so (built by ``rl_post_linear_gb300.build``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("librlk.so not found at %s: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`" % path)
    lib = ctypes.CDLL(path)
    lib.rlk_linear_logp_fwd_workspace_bytes.restype = _sz
    lib.rlk_linear_logp_fwd_workspace_bytes.argtypes = [_i64, _i64, _i64]
    lib.rlk_linear_logp_bwd_workspace_bytes.restype = _sz
    lib.rlk_linear_logp_bwd_workspace_bytes.argtypes = [_i64, _i64, _i64]
    lib.rlk_dlogp_audit_workspace_bytes.restype = _sz
    lib.rlk_dlogp_audit_workspace_bytes.argtypes = [_i64]
    lib.rlk_linear_logp_fwd.restype = ctypes.c_int
    lib.rlk_linear_logp_fwd.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_double,
                                        _vp, _vp, _vp, _sz, _vp, _vp]
    lib.rlk_linear_logp_bwd.restype = ctypes.c_int
    lib.rlk_linear_logp_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64,
                                        ctypes.c_double, _vp, _vp, _vp, _sz, _vp, _vp]
    lib.rlk_dlogp_audit.restype = ctypes.c_int
    lib.rlk_dlogp_audit.argtypes = [_vp, _vp, _vp, _i64, _vp, _vp, _sz, _vp]
    lib.rlk_dlogp_audit_noalloc.restype = ctypes.c_int
    lib.rlk_dlogp_audit_noalloc.argtypes = [_vp, _vp, _vp, _i64, _vp, _vp]
    lib.rlk_contract_string.restype = ctypes.c_char_p
    lib.rlk_contract_string.argtypes = []
    lib.rlk_status_string.restype = ctypes.c_char_p
    lib.rlk_status_string.argtypes = [ctypes.c_int]
    _lib = lib
    return lib


def declared_functions(header: str = HEADER_PATH):
    """Names of the functions declared in include/rlk.h."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rlk_[a-z0-9_]+)\s*\(", text)))


def status_string(status: int) -> str:
    return load().rlk_status_string(int(status)).decode()


def rlk_contract_string() -> str:
    return load().rlk_contract_string().decode()


def rlk_linear_logp_fwd_workspace_bytes(N: int, H: int, V: int) -> int:
    return int(load().rlk_linear_logp_fwd_workspace_bytes(N, H, V))


def rlk_linear_logp_bwd_workspace_bytes(N: int, H: int, V: int) -> int:
    return int(load().rlk_linear_logp_bwd_workspace_bytes(N, H, V))


def rlk_dlogp_audit_workspace_bytes(N: int) -> int:
    return int(load().rlk_dlogp_audit_workspace_bytes(N))


# ----------------------------------------------------------------------------- marshalling

def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _need(t, dtype, name, shape=None):
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def _check(fn, status):
    if status != RLK_OK:
        raise RlkError(fn, status)


def rlk_linear_logp_fwd(hidden, weight, targets, active_mask, temperature, logp_out, lse_out,
                        workspace, device_error_word=None, stream=None):
    """Enqueue the forward; see include/rlk.h.  All tensors are caller-allocated on the GPU."""
    n, h = hidden.shape
    v = weight.shape[0]
    _need(hidden, torch.bfloat16, "hidden")
    _need(weight, torch.bfloat16, "weight", (v, h))
    _need(targets, torch.int64, "targets", (n,))
    if active_mask is not None:
        _need(active_mask, torch.uint8, "active_mask", (n,))
    _need(logp_out, torch.float32, "logp_out", (n,))
    if lse_out is not None:
        _need(lse_out, torch.float32, "lse_out", (n,))
    _need(workspace, torch.uint8, "workspace")
    st = load().rlk_linear_logp_fwd(_ptr(hidden), _ptr(weight), _ptr(targets), _ptr(active_mask),
                                    n, h, v, float(temperature), _ptr(logp_out), _ptr(lse_out),
                                    _ptr(workspace), workspace.numel(), _ptr(device_error_word),
                                    _stream(stream))
    _check("rlk_linear_logp_fwd", st)


def rlk_linear_logp_bwd(hidden, weight, targets, active_mask, grad_logp, lse, temperature,
                        dhidden, dweight, workspace, device_error_word=None, stream=None):
    """Enqueue the backward; see include/rlk.h."""
    n, h = hidden.shape
    v = weight.shape[0]
    _need(hidden, torch.bfloat16, "hidden")
    _need(weight, torch.bfloat16, "weight", (v, h))
    _need(targets, torch.int64, "targets", (n,))
    if active_mask is not None:
        _need(active_mask, torch.uint8, "active_mask", (n,))
    _need(grad_logp, torch.float32, "grad_logp", (n,))
    _need(lse, torch.float32, "lse", (n,))
    _need(dhidden, torch.bfloat16, "dhidden", (n, h))
    _need(dweight, torch.bfloat16, "dweight", (v, h))
    _need(workspace, torch.uint8, "workspace")
    st = load().rlk_linear_logp_bwd(_ptr(hidden), _ptr(weight), _ptr(targets), _ptr(active_mask),
                                    _ptr(grad_logp), _ptr(lse), n, h, v, float(temperature),
                                    _ptr(dhidden), _ptr(dweight), _ptr(workspace),
                                    workspace.numel(), _ptr(device_error_word), _stream(stream))
    _check("rlk_linear_logp_bwd", st)


def rlk_dlogp_audit(logp_new, logp_old, active_mask, result, workspace, stream=None):
    """Enqueue the audit; ``result`` is a uint8 CUDA tensor of AUDIT_RESULT_BYTES bytes."""
    n = logp_new.shape[0]
    _need(logp_new, torch.float32, "logp_new", (n,))
    _need(logp_old, torch.float32, "logp_old", (n,))
    if active_mask is not None:
        _need(active_mask, torch.uint8, "active_mask", (n,))
    _need(result, torch.uint8, "result", (AUDIT_RESULT_BYTES,))
    _need(workspace, torch.uint8, "workspace")
    st = load().rlk_dlogp_audit(_ptr(logp_new), _ptr(logp_old), _ptr(active_mask), n,
                                _ptr(result), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("rlk_dlogp_audit", st)


def rlk_dlogp_audit_noalloc(logp_new, logp_old, active_mask, result, stream=None):
    """The audit without a workspace, for callers that cannot allocate device memory (a
    rollout engine that reserved nearly all of it up front, a hook limited to the tensors it
    is handed).  Scratch is a fixed 1.25 MiB array inside the library, shared by every call:
    N <= RLK_AUDIT_NOALLOC_MAX_N, and calls must not overlap on the GPU.  The first call on
    a device looks the array's address up, so make it before any stream capture."""
    n = logp_new.shape[0]
    _need(logp_new, torch.float32, "logp_new", (n,))
    _need(logp_old, torch.float32, "logp_old", (n,))
    if active_mask is not None:
        _need(active_mask, torch.uint8, "active_mask", (n,))
    _need(result, torch.uint8, "result", (AUDIT_RESULT_BYTES,))
    st = load().rlk_dlogp_audit_noalloc(_ptr(logp_new), _ptr(logp_old), _ptr(active_mask), n,
                                        _ptr(result), _stream(stream))
    _check("rlk_dlogp_audit_noalloc", st)


# ----------------------------------------------------------------------------- conveniences

def _workspace(nbytes, device):
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def linear_logp_fwd(hidden, weight, targets, active_mask=None, temperature=1.0, error_word=None):
    """(logp[N], lse[N]) fp32, allocated with torch on the inputs' device."""
    n, h = hidden.shape
    v = weight.shape[0]
    logp = torch.empty(n, dtype=torch.float32, device=hidden.device)
    lse = torch.empty(n, dtype=torch.float32, device=hidden.device)
    ws = _workspace(rlk_linear_logp_fwd_workspace_bytes(n, h, v), hidden.device)
    rlk_linear_logp_fwd(hidden, weight, targets, active_mask, temperature, logp, lse, ws,
                        error_word)
    return logp, lse


def linear_logp_bwd(hidden, weight, targets, active_mask, grad_logp, lse, temperature=1.0,
                    error_word=None):
    """(dhidden[N,H], dweight[V,H]) bf16, allocated with torch."""
    n, h = hidden.shape
    v = weight.shape[0]
    dh = torch.empty_like(hidden)
    dw = torch.empty_like(weight)
    ws = _workspace(rlk_linear_logp_bwd_workspace_bytes(n, h, v), hidden.device)
    rlk_linear_logp_bwd(hidden, weight, targets, active_mask, grad_logp, lse, temperature, dh, dw,
                        ws, error_word)
    return dh, dw


def audit_result_to_dict(raw: torch.Tensor) -> dict:
    r = AuditResult.from_buffer_copy(bytes(raw.cpu().numpy().tobytes()))
    return {f: getattr(r, f) for f, _ in AuditResult._fields_}


def dlogp_audit(logp_new, logp_old, active_mask=None):
    """Audit dict (synchronises to read the result back)."""
    n = logp_new.shape[0]
    res = torch.empty(AUDIT_RESULT_BYTES, dtype=torch.uint8, device=logp_new.device)
    ws = _workspace(rlk_dlogp_audit_workspace_bytes(n), logp_new.device)
    rlk_dlogp_audit(logp_new, logp_old, active_mask, res, ws)
    return audit_result_to_dict(res)


class LinearLogp(torch.autograd.Function):
    """logp = LinearLogp.apply(hidden, weight, targets, active_mask, temperature)."""

    @staticmethod
    def forward(ctx, hidden, weight, targets, active_mask, temperature):
        logp, lse = linear_logp_fwd(hidden, weight, targets, active_mask, temperature)
        ctx.save_for_backward(hidden, weight, targets, active_mask, lse)
        ctx.temperature = temperature
        return logp

    @staticmethod
    def backward(ctx, grad_logp):
        hidden, weight, targets, active_mask, lse = ctx.saved_tensors
        dh, dw = linear_logp_bwd(hidden, weight, targets, active_mask,
                                 grad_logp.float().contiguous(), lse, ctx.temperature)
        return dh, dw, None, None, None


def linear_logp(hidden, weight, targets, active_mask=None, temperature=1.0):
    return LinearLogp.apply(hidden, weight, targets, active_mask, temperature)
