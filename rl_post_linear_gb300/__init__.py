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
RLK_DEVERR_ROW_RANGE = 0x4
RLK_DTYPE_F32, RLK_DTYPE_BF16 = 0, 1
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


class AuditExtResult(ctypes.Structure):
    """Mirror of rlk_audit_ext_t."""
    _fields_ = [(n, ctypes.c_int64) for n in ("active_count", "argmax_index", "argmax_seq",
                                               "argmax_pos", "clip_count")] + \
               [(n, ctypes.c_double) for n in ("mean_dlogp", "mean_abs_dlogp", "mean_ratio",
                                                "approx_kl")] + \
               [(n, ctypes.c_float) for n in ("max_abs_dlogp", "p50_abs_dlogp", "p90_abs_dlogp",
                                               "p99_abs_dlogp", "clipfrac")] + \
               [("error_flags", ctypes.c_uint32)]


AUDIT_EXT_RESULT_BYTES = ctypes.sizeof(AuditExtResult)


class GrpoResult(ctypes.Structure):
    """Mirror of rlk_grpo_result_t."""
    _fields_ = [
        ("active_count", ctypes.c_int64),
        ("clipped_count", ctypes.c_int64),
        ("outside_count", ctypes.c_int64),
        ("loss", ctypes.c_double),
        ("mean_ratio", ctypes.c_double),
    ]


GRPO_RESULT_BYTES = ctypes.sizeof(GrpoResult)


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
    lib.rlk_linear_logp_entropy_bwd_workspace_bytes.restype = _sz
    lib.rlk_linear_logp_entropy_bwd_workspace_bytes.argtypes = [_i64, _i64, _i64]
    lib.rlk_dlogp_audit_workspace_bytes.restype = _sz
    lib.rlk_dlogp_audit_workspace_bytes.argtypes = [_i64]
    lib.rlk_linear_logp_fwd.restype = ctypes.c_int
    lib.rlk_linear_logp_fwd.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_double,
                                        _vp, _vp, _vp, _sz, _vp, _vp]
    lib.rlk_linear_logp_bwd.restype = ctypes.c_int
    lib.rlk_linear_logp_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64,
                                        ctypes.c_double, _vp, _vp, _vp, _sz, _vp, _vp]
    lib.rlk_linear_logp_entropy_fwd.restype = ctypes.c_int
    lib.rlk_linear_logp_entropy_fwd.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64,
                                                ctypes.c_double, _vp, _vp, _vp, _vp, _sz, _vp,
                                                _vp]
    lib.rlk_linear_kl_fwd_workspace_bytes.restype = _sz
    lib.rlk_linear_kl_fwd_workspace_bytes.argtypes = [_i64, _i64]
    lib.rlk_linear_kl_fwd.restype = ctypes.c_int
    lib.rlk_linear_kl_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                      ctypes.c_double, ctypes.c_double, _vp, _vp, _vp, _vp, _vp,
                                      _vp, _sz, _vp, _vp]
    lib.rlk_linear_kl_bwd_workspace_bytes.restype = _sz
    lib.rlk_linear_kl_bwd_workspace_bytes.argtypes = [_i64, _i64, _i64]
    lib.rlk_linear_kl_bwd.restype = ctypes.c_int
    lib.rlk_linear_kl_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64,
                                      _i64, _i64, _i64, ctypes.c_double, ctypes.c_double, _vp,
                                      _vp, _vp, _sz, _vp, _vp]
    lib.rlk_linear_logp_bwd_shard.restype = ctypes.c_int
    lib.rlk_linear_logp_bwd_shard.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64,
                                              _i64, _i64, ctypes.c_double, _vp, _vp, _vp, _sz,
                                              _vp, _vp]
    lib.rlk_linear_logp_dh_merge.restype = ctypes.c_int
    lib.rlk_linear_logp_dh_merge.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp]
    lib.rlk_linear_logp_bwd_dw_partial.restype = ctypes.c_int
    lib.rlk_linear_logp_bwd_dw_partial.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                                                   _i64, ctypes.c_double, _vp, _vp, _vp, _sz,
                                                   _vp, _vp]
    lib.rlk_linear_logp_dw_merge.restype = ctypes.c_int
    lib.rlk_linear_logp_dw_merge.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp]
    lib.rlk_linear_logp_entropy_bwd.restype = ctypes.c_int
    lib.rlk_linear_logp_entropy_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64,
                                                _i64, _i64, ctypes.c_double, _vp, _vp, _vp, _sz,
                                                _vp, _vp]
    lib.rlk_dlogp_audit.restype = ctypes.c_int
    lib.rlk_dlogp_audit.argtypes = [_vp, _vp, _vp, _i64, _vp, _vp, _sz, _vp]
    lib.rlk_linear_logp_num_partials.restype = _i64
    lib.rlk_linear_logp_num_partials.argtypes = [_i64]
    lib.rlk_linear_logp_fwd_shard.restype = ctypes.c_int
    lib.rlk_linear_logp_fwd_shard.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                              ctypes.c_double, _vp, _vp, _vp, _vp]
    lib.rlk_linear_logp_merge.restype = ctypes.c_int
    lib.rlk_linear_logp_merge.argtypes = [_vp, _i64, _vp, _vp, _vp, _i64, _i64, ctypes.c_double,
                                          _vp, _vp, _vp, _vp]
    lib.rlk_logp_from_logits.restype = ctypes.c_int
    lib.rlk_logp_from_logits.argtypes = [_vp, ctypes.c_int32, _i64, _i64, _i64, _vp, _i64, _vp,
                                         _vp, ctypes.c_double, _vp, _vp, _vp, _vp]
    lib.rlk_grpo_clip_loss_workspace_bytes.restype = _sz
    lib.rlk_grpo_clip_loss_workspace_bytes.argtypes = [_i64]
    lib.rlk_grpo_clip_loss.restype = ctypes.c_int
    lib.rlk_grpo_clip_loss.argtypes = [_vp, _vp, _vp, _vp, _i64, ctypes.c_double, ctypes.c_double,
                                       ctypes.c_double, _vp, _vp, _vp, _sz, _vp]
    lib.rlk_dlogp_audit_ext_workspace_bytes.restype = _sz
    lib.rlk_dlogp_audit_ext_workspace_bytes.argtypes = [_i64]
    lib.rlk_dlogp_audit_ext.restype = ctypes.c_int
    lib.rlk_dlogp_audit_ext.argtypes = [_vp, _vp, _vp, _i64, _vp, _i64, ctypes.c_double, _vp,
                                        _vp, _sz, _vp]
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


def rlk_linear_logp_entropy_bwd_workspace_bytes(N: int, H: int, V: int) -> int:
    return int(load().rlk_linear_logp_entropy_bwd_workspace_bytes(N, H, V))


def rlk_dlogp_audit_workspace_bytes(N: int) -> int:
    return int(load().rlk_dlogp_audit_workspace_bytes(N))


def rlk_linear_logp_num_partials(V_local: int) -> int:
    return int(load().rlk_linear_logp_num_partials(V_local))


def rlk_dlogp_audit_ext_workspace_bytes(N: int) -> int:
    return int(load().rlk_dlogp_audit_ext_workspace_bytes(N))


def rlk_grpo_clip_loss_workspace_bytes(N: int) -> int:
    return int(load().rlk_grpo_clip_loss_workspace_bytes(N))


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


def rlk_linear_logp_entropy_fwd(hidden, weight, targets, active_mask, temperature, logp_out,
                                lse_out, entropy_out, workspace, device_error_word=None,
                                stream=None):
    """Forward with the softmax entropy as a second output; see include/rlk.h."""
    n, h = hidden.shape
    v = weight.shape[0]
    _need(hidden, torch.bfloat16, "hidden")
    _need(weight, torch.bfloat16, "weight", (v, h))
    _need(targets, torch.int64, "targets", (n,))
    if active_mask is not None:
        _need(active_mask, torch.uint8, "active_mask", (n,))
    for t, name in ((logp_out, "logp_out"), (entropy_out, "entropy_out")):
        _need(t, torch.float32, name, (n,))
    if lse_out is not None:
        _need(lse_out, torch.float32, "lse_out", (n,))
    _need(workspace, torch.uint8, "workspace")
    st = load().rlk_linear_logp_entropy_fwd(_ptr(hidden), _ptr(weight), _ptr(targets),
                                            _ptr(active_mask), n, h, v, float(temperature),
                                            _ptr(logp_out), _ptr(lse_out), _ptr(entropy_out),
                                            _ptr(workspace), workspace.numel(),
                                            _ptr(device_error_word), _stream(stream))
    _check("rlk_linear_logp_entropy_fwd", st)


def rlk_linear_logp_entropy_bwd(hidden, weight, targets, active_mask, grad_logp, grad_entropy,
                                lse, entropy, temperature, dhidden, dweight, workspace,
                                device_error_word=None, stream=None):
    """Backward of sum g logp + sum gH entropy; see include/rlk.h."""
    n, h = hidden.shape
    v = weight.shape[0]
    _need(hidden, torch.bfloat16, "hidden")
    _need(weight, torch.bfloat16, "weight", (v, h))
    _need(targets, torch.int64, "targets", (n,))
    if active_mask is not None:
        _need(active_mask, torch.uint8, "active_mask", (n,))
    for t, name in ((grad_logp, "grad_logp"), (grad_entropy, "grad_entropy"), (lse, "lse"),
                    (entropy, "entropy")):
        _need(t, torch.float32, name, (n,))
    _need(dhidden, torch.bfloat16, "dhidden", (n, h))
    _need(dweight, torch.bfloat16, "dweight", (v, h))
    _need(workspace, torch.uint8, "workspace")
    st = load().rlk_linear_logp_entropy_bwd(_ptr(hidden), _ptr(weight), _ptr(targets),
                                            _ptr(active_mask), _ptr(grad_logp),
                                            _ptr(grad_entropy), _ptr(lse), _ptr(entropy), n, h,
                                            v, float(temperature), _ptr(dhidden), _ptr(dweight),
                                            _ptr(workspace), workspace.numel(),
                                            _ptr(device_error_word), _stream(stream))
    _check("rlk_linear_logp_entropy_bwd", st)


def rlk_linear_kl_fwd_workspace_bytes(N: int, V: int) -> int:
    return int(load().rlk_linear_kl_fwd_workspace_bytes(N, V))


def rlk_linear_kl_fwd(hidden, weight, hidden_ref, weight_ref, targets, active_mask, temperature,
                      temperature_ref, kl_out, kl_rev_out, lse_out, lse_ref_out, logp_out,
                      workspace, device_error_word=None, stream=None):
    """Full-vocabulary KL of the policy head against a reference head; see include/rlk.h."""
    n, h = hidden.shape
    v = weight.shape[0]
    hr = hidden_ref.shape[1]
    _need(hidden, torch.bfloat16, "hidden")
    _need(weight, torch.bfloat16, "weight", (v, h))
    _need(hidden_ref, torch.bfloat16, "hidden_ref", (n, hr))
    _need(weight_ref, torch.bfloat16, "weight_ref", (v, hr))
    if targets is not None:
        _need(targets, torch.int64, "targets", (n,))
    if active_mask is not None:
        _need(active_mask, torch.uint8, "active_mask", (n,))
    _need(kl_out, torch.float32, "kl_out", (n,))
    for t, name in ((kl_rev_out, "kl_rev_out"), (lse_out, "lse_out"),
                    (lse_ref_out, "lse_ref_out"), (logp_out, "logp_out")):
        if t is not None:
            _need(t, torch.float32, name, (n,))
    _need(workspace, torch.uint8, "workspace")
    st = load().rlk_linear_kl_fwd(_ptr(hidden), _ptr(weight), _ptr(hidden_ref), _ptr(weight_ref),
                                  _ptr(targets), _ptr(active_mask), n, h, hr, v,
                                  float(temperature), float(temperature_ref), _ptr(kl_out),
                                  _ptr(kl_rev_out), _ptr(lse_out), _ptr(lse_ref_out),
                                  _ptr(logp_out), _ptr(workspace), workspace.numel(),
                                  _ptr(device_error_word), _stream(stream))
    _check("rlk_linear_kl_fwd", st)


def rlk_linear_kl_bwd_workspace_bytes(N: int, H: int, V: int) -> int:
    return int(load().rlk_linear_kl_bwd_workspace_bytes(N, H, V))


def rlk_linear_kl_bwd(hidden, weight, hidden_ref, weight_ref, active_mask, grad_kl, grad_kl_rev,
                      lse, lse_ref, kl, temperature, temperature_ref, dhidden, dweight,
                      workspace, device_error_word=None, stream=None):
    """Backward of sum g kl + sum gr kl_rev for the policy head; see include/rlk.h."""
    n, h = hidden.shape
    v = weight.shape[0]
    hr = hidden_ref.shape[1]
    _need(hidden, torch.bfloat16, "hidden")
    _need(weight, torch.bfloat16, "weight", (v, h))
    _need(hidden_ref, torch.bfloat16, "hidden_ref", (n, hr))
    _need(weight_ref, torch.bfloat16, "weight_ref", (v, hr))
    if active_mask is not None:
        _need(active_mask, torch.uint8, "active_mask", (n,))
    for t, name in ((grad_kl, "grad_kl"), (grad_kl_rev, "grad_kl_rev"), (kl, "kl")):
        if t is not None:
            _need(t, torch.float32, name, (n,))
    _need(lse, torch.float32, "lse", (n,))
    _need(lse_ref, torch.float32, "lse_ref", (n,))
    _need(dhidden, torch.bfloat16, "dhidden", (n, h))
    _need(dweight, torch.bfloat16, "dweight", (v, h))
    _need(workspace, torch.uint8, "workspace")
    st = load().rlk_linear_kl_bwd(_ptr(hidden), _ptr(weight), _ptr(hidden_ref), _ptr(weight_ref),
                                  _ptr(active_mask), _ptr(grad_kl), _ptr(grad_kl_rev), _ptr(lse),
                                  _ptr(lse_ref), _ptr(kl), n, h, hr, v, float(temperature),
                                  float(temperature_ref), _ptr(dhidden), _ptr(dweight),
                                  _ptr(workspace), workspace.numel(), _ptr(device_error_word),
                                  _stream(stream))
    _check("rlk_linear_kl_bwd", st)


def rlk_linear_logp_bwd_shard(hidden, weight_shard, targets, active_mask, grad_logp, lse,
                              vocab_start, vocab_size, temperature, dhidden_partial,
                              dweight_shard, workspace, device_error_word=None, stream=None):
    """One vocab block's fp32 dh partial and dW rows; see include/rlk.h."""
    n, h = hidden.shape
    v_local = weight_shard.shape[0]
    _need(hidden, torch.bfloat16, "hidden")
    _need(weight_shard, torch.bfloat16, "weight_shard", (v_local, h))
    _need(targets, torch.int64, "targets", (n,))
    if active_mask is not None:
        _need(active_mask, torch.uint8, "active_mask", (n,))
    _need(grad_logp, torch.float32, "grad_logp", (n,))
    _need(lse, torch.float32, "lse", (n,))
    _need(dhidden_partial, torch.float32, "dhidden_partial", (n, h))
    _need(dweight_shard, torch.bfloat16, "dweight_shard", (v_local, h))
    _need(workspace, torch.uint8, "workspace")
    st = load().rlk_linear_logp_bwd_shard(_ptr(hidden), _ptr(weight_shard), _ptr(targets),
                                          _ptr(active_mask), _ptr(grad_logp), _ptr(lse), n, h,
                                          v_local, int(vocab_start), int(vocab_size),
                                          float(temperature), _ptr(dhidden_partial),
                                          _ptr(dweight_shard), _ptr(workspace), workspace.numel(),
                                          _ptr(device_error_word), _stream(stream))
    _check("rlk_linear_logp_bwd_shard", st)


def rlk_linear_logp_dh_merge(dh_partials, dhidden, stream=None):
    """dhidden = bf16(sum over the leading axis of dh_partials [k, N, H] fp32), ascending."""
    k, n, h = dh_partials.shape
    _need(dh_partials, torch.float32, "dh_partials")
    _need(dhidden, torch.bfloat16, "dhidden", (n, h))
    st = load().rlk_linear_logp_dh_merge(_ptr(dh_partials), k, n, h, _ptr(dhidden),
                                         _stream(stream))
    _check("rlk_linear_logp_dh_merge", st)


def rlk_linear_logp_bwd_dw_partial(hidden, weight, targets, active_mask, grad_logp, lse,
                                   temperature, dhidden, dweight_partial, workspace,
                                   device_error_word=None, stream=None):
    """One data-parallel rank's backward: bf16 dhidden and an unrounded fp32 dW partial."""
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
    _need(dweight_partial, torch.float32, "dweight_partial", (v, h))
    _need(workspace, torch.uint8, "workspace")
    st = load().rlk_linear_logp_bwd_dw_partial(_ptr(hidden), _ptr(weight), _ptr(targets),
                                               _ptr(active_mask), _ptr(grad_logp), _ptr(lse), n,
                                               h, v, float(temperature), _ptr(dhidden),
                                               _ptr(dweight_partial), _ptr(workspace),
                                               workspace.numel(), _ptr(device_error_word),
                                               _stream(stream))
    _check("rlk_linear_logp_bwd_dw_partial", st)


def rlk_linear_logp_dw_merge(dw_partials, dweight, stream=None):
    """dweight = bf16(sum over the leading axis of dw_partials [k, V, H] fp32), ascending."""
    k, v, h = dw_partials.shape
    _need(dw_partials, torch.float32, "dw_partials")
    _need(dweight, torch.bfloat16, "dweight", (v, h))
    st = load().rlk_linear_logp_dw_merge(_ptr(dw_partials), k, v, h, _ptr(dweight),
                                         _stream(stream))
    _check("rlk_linear_logp_dw_merge", st)


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


def rlk_dlogp_audit_ext(logp_new, logp_old, active_mask, seq_offsets, clip_eps, result,
                        workspace, stream=None):
    """Extended diagnostics; ``result`` is a uint8 CUDA tensor of AUDIT_EXT_RESULT_BYTES bytes,
    ``seq_offsets`` an int64 CUDA tensor [num_seqs + 1] or None.  See include/rlk.h."""
    n = logp_new.shape[0]
    _need(logp_new, torch.float32, "logp_new", (n,))
    _need(logp_old, torch.float32, "logp_old", (n,))
    if active_mask is not None:
        _need(active_mask, torch.uint8, "active_mask", (n,))
    num_seqs = 0
    if seq_offsets is not None:
        _need(seq_offsets, torch.int64, "seq_offsets")
        num_seqs = seq_offsets.numel() - 1
    _need(result, torch.uint8, "result", (AUDIT_EXT_RESULT_BYTES,))
    _need(workspace, torch.uint8, "workspace")
    st = load().rlk_dlogp_audit_ext(_ptr(logp_new), _ptr(logp_old), _ptr(active_mask), n,
                                    _ptr(seq_offsets), num_seqs, float(clip_eps), _ptr(result),
                                    _ptr(workspace), workspace.numel(), _stream(stream))
    _check("rlk_dlogp_audit_ext", st)


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


def rlk_linear_logp_fwd_shard(hidden, weight_shard, targets, active_mask, vocab_start,
                              temperature, partials_out, target_logit_out,
                              device_error_word=None, stream=None):
    """Partials of one vocab block; see include/rlk.h.  partials_out: float32
    [num_partials(V_local), N, 2] (or any contiguous view of it)."""
    n, h = hidden.shape
    v_local = weight_shard.shape[0]
    _need(hidden, torch.bfloat16, "hidden")
    _need(weight_shard, torch.bfloat16, "weight_shard", (v_local, h))
    _need(targets, torch.int64, "targets", (n,))
    if active_mask is not None:
        _need(active_mask, torch.uint8, "active_mask", (n,))
    _need(partials_out, torch.float32, "partials_out")
    if partials_out.numel() < rlk_linear_logp_num_partials(v_local) * n * 2:
        raise ValueError("partials_out is too small")
    _need(target_logit_out, torch.float32, "target_logit_out", (n,))
    st = load().rlk_linear_logp_fwd_shard(_ptr(hidden), _ptr(weight_shard), _ptr(targets),
                                          _ptr(active_mask), n, h, v_local, int(vocab_start),
                                          float(temperature), _ptr(partials_out),
                                          _ptr(target_logit_out), _ptr(device_error_word),
                                          _stream(stream))
    _check("rlk_linear_logp_fwd_shard", st)


def rlk_linear_logp_merge(partials, num_partials, target_logit, targets, active_mask, vocab_size,
                          temperature, logp_out, lse_out, device_error_word=None, stream=None):
    """Fixed-order merge of block partials (global chunk order); see include/rlk.h."""
    n = targets.shape[0]
    _need(partials, torch.float32, "partials")
    if partials.numel() < num_partials * n * 2:
        raise ValueError("partials is too small")
    _need(target_logit, torch.float32, "target_logit", (n,))
    _need(targets, torch.int64, "targets", (n,))
    if active_mask is not None:
        _need(active_mask, torch.uint8, "active_mask", (n,))
    _need(logp_out, torch.float32, "logp_out", (n,))
    if lse_out is not None:
        _need(lse_out, torch.float32, "lse_out", (n,))
    st = load().rlk_linear_logp_merge(_ptr(partials), int(num_partials), _ptr(target_logit),
                                      _ptr(targets), _ptr(active_mask), n, int(vocab_size),
                                      float(temperature), _ptr(logp_out), _ptr(lse_out),
                                      _ptr(device_error_word), _stream(stream))
    _check("rlk_linear_logp_merge", st)


def rlk_logp_from_logits(logits, rows, targets, active_mask, temperature, logp_out, lse_out,
                         device_error_word=None, stream=None):
    """Score rows of existing logits [N, V] (fp32 or bf16, rows contiguous, any row stride);
    rows = None scores all N rows.  See include/rlk.h."""
    if logits.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("logits must be float32 or bfloat16")
    if not logits.is_cuda or logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be a 2-D CUDA tensor with contiguous rows")
    n, v = logits.shape
    _need(targets, torch.int64, "targets", (n,))
    if active_mask is not None:
        _need(active_mask, torch.uint8, "active_mask", (n,))
    m = n if rows is None else rows.shape[0]
    if rows is not None:
        _need(rows, torch.int64, "rows", (m,))
    _need(logp_out, torch.float32, "logp_out", (m,))
    if lse_out is not None:
        _need(lse_out, torch.float32, "lse_out", (m,))
    dt = RLK_DTYPE_F32 if logits.dtype == torch.float32 else RLK_DTYPE_BF16
    st = load().rlk_logp_from_logits(_ptr(logits), dt, n, v, logits.stride(0), _ptr(rows), m,
                                     _ptr(targets), _ptr(active_mask), float(temperature),
                                     _ptr(logp_out), _ptr(lse_out), _ptr(device_error_word),
                                     _stream(stream))
    _check("rlk_logp_from_logits", st)


def rlk_grpo_clip_loss(logp_new, logp_old, advantages, active_mask, eps_low, eps_high,
                       loss_scale, grad_out, result, workspace, stream=None):
    """Enqueue the clipped-ratio loss fragment; see include/rlk.h."""
    n = logp_new.shape[0]
    _need(logp_new, torch.float32, "logp_new", (n,))
    _need(logp_old, torch.float32, "logp_old", (n,))
    _need(advantages, torch.float32, "advantages", (n,))
    if active_mask is not None:
        _need(active_mask, torch.uint8, "active_mask", (n,))
    _need(grad_out, torch.float32, "grad_out", (n,))
    _need(result, torch.uint8, "result", (GRPO_RESULT_BYTES,))
    _need(workspace, torch.uint8, "workspace")
    st = load().rlk_grpo_clip_loss(_ptr(logp_new), _ptr(logp_old), _ptr(advantages),
                                   _ptr(active_mask), n, float(eps_low), float(eps_high),
                                   float(loss_scale), _ptr(grad_out), _ptr(result),
                                   _ptr(workspace), workspace.numel(), _stream(stream))
    _check("rlk_grpo_clip_loss", st)


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


def linear_logp_entropy_fwd(hidden, weight, targets, active_mask=None, temperature=1.0,
                            error_word=None):
    """(logp[N], lse[N], entropy[N]) fp32."""
    n, h = hidden.shape
    v = weight.shape[0]
    logp, lse, ent = (torch.empty(n, dtype=torch.float32, device=hidden.device) for _ in range(3))
    ws = _workspace(rlk_linear_logp_fwd_workspace_bytes(n, h, v), hidden.device)
    rlk_linear_logp_entropy_fwd(hidden, weight, targets, active_mask, temperature, logp, lse, ent,
                                ws, error_word)
    return logp, lse, ent


def linear_logp_entropy_bwd(hidden, weight, targets, active_mask, grad_logp, grad_entropy, lse,
                            entropy, temperature=1.0, error_word=None):
    """(dhidden[N,H], dweight[V,H]) bf16."""
    n, h = hidden.shape
    v = weight.shape[0]
    dh = torch.empty_like(hidden)
    dw = torch.empty_like(weight)
    ws = _workspace(rlk_linear_logp_entropy_bwd_workspace_bytes(n, h, v), hidden.device)
    rlk_linear_logp_entropy_bwd(hidden, weight, targets, active_mask, grad_logp, grad_entropy,
                                lse, entropy, temperature, dh, dw, ws, error_word)
    return dh, dw


def linear_kl_fwd(hidden, weight, hidden_ref, weight_ref, active_mask=None, temperature=1.0,
                  temperature_ref=None, targets=None, error_word=None):
    """(kl, kl_rev, lse, lse_ref, logp or None), each fp32 [N]: KL(p || q) and KL(q || p)
    between the policy head (hidden, weight, temperature) and the reference head."""
    n = hidden.shape[0]
    v = weight.shape[0]
    temperature_ref = temperature if temperature_ref is None else temperature_ref
    outs = [torch.empty(n, dtype=torch.float32, device=hidden.device) for _ in range(4)]
    logp = None if targets is None else torch.empty(n, dtype=torch.float32, device=hidden.device)
    ws = _workspace(rlk_linear_kl_fwd_workspace_bytes(n, v), hidden.device)
    rlk_linear_kl_fwd(hidden, weight, hidden_ref, weight_ref, targets, active_mask, temperature,
                      temperature_ref, *outs, logp, ws, error_word)
    return (*outs, logp)


def linear_kl_bwd(hidden, weight, hidden_ref, weight_ref, active_mask, grad_kl, grad_kl_rev,
                  lse, lse_ref, kl, temperature=1.0, temperature_ref=None, error_word=None):
    """(dhidden[N,H], dweight[V,H]) bf16 of sum g kl + sum gr kl_rev (policy head only)."""
    n, h = hidden.shape
    v = weight.shape[0]
    temperature_ref = temperature if temperature_ref is None else temperature_ref
    dh = torch.empty_like(hidden)
    dw = torch.empty_like(weight)
    ws = _workspace(rlk_linear_kl_bwd_workspace_bytes(n, h, v), hidden.device)
    rlk_linear_kl_bwd(hidden, weight, hidden_ref, weight_ref, active_mask, grad_kl, grad_kl_rev,
                      lse, lse_ref, kl, temperature, temperature_ref, dh, dw, ws, error_word)
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


def grpo_clip_loss(logp_new, logp_old, advantages, active_mask, eps_low, eps_high, loss_scale):
    """(grad[N] fp32, result dict); synchronises to read the result back."""
    n = logp_new.shape[0]
    grad = torch.empty(n, dtype=torch.float32, device=logp_new.device)
    res = torch.empty(GRPO_RESULT_BYTES, dtype=torch.uint8, device=logp_new.device)
    ws = _workspace(rlk_grpo_clip_loss_workspace_bytes(n), logp_new.device)
    rlk_grpo_clip_loss(logp_new, logp_old, advantages, active_mask, eps_low, eps_high, loss_scale,
                       grad, res, ws)
    r = GrpoResult.from_buffer_copy(bytes(res.cpu().numpy().tobytes()))
    return grad, {f: getattr(r, f) for f, _ in GrpoResult._fields_}


def logp_from_logits(logits, targets, active_mask=None, temperature=1.0, rows=None,
                     error_word=None):
    """(logp[M], lse[M]) fp32 for the selected rows of existing logits."""
    m = logits.shape[0] if rows is None else rows.shape[0]
    logp = torch.empty(m, dtype=torch.float32, device=logits.device)
    lse = torch.empty(m, dtype=torch.float32, device=logits.device)
    rlk_logp_from_logits(logits, rows, targets, active_mask, temperature, logp, lse, error_word)
    return logp, lse


def dlogp_audit_ext(logp_new, logp_old, active_mask=None, seq_offsets=None, clip_eps=0.2):
    """Extended diagnostics dict (synchronises to read the result back)."""
    n = logp_new.shape[0]
    res = torch.empty(AUDIT_EXT_RESULT_BYTES, dtype=torch.uint8, device=logp_new.device)
    ws = _workspace(rlk_dlogp_audit_ext_workspace_bytes(n), logp_new.device)
    rlk_dlogp_audit_ext(logp_new, logp_old, active_mask, seq_offsets, clip_eps, res, ws)
    r = AuditExtResult.from_buffer_copy(bytes(res.cpu().numpy().tobytes()))
    return {f: getattr(r, f) for f, _ in AuditExtResult._fields_}


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


class LinearLogpEntropy(torch.autograd.Function):
    """(logp, entropy) = LinearLogpEntropy.apply(hidden, weight, targets, active_mask, T)."""

    @staticmethod
    def forward(ctx, hidden, weight, targets, active_mask, temperature):
        logp, lse, ent = linear_logp_entropy_fwd(hidden, weight, targets, active_mask, temperature)
        ctx.save_for_backward(hidden, weight, targets, active_mask, lse, ent)
        ctx.temperature = temperature
        return logp, ent

    @staticmethod
    def backward(ctx, grad_logp, grad_entropy):
        hidden, weight, targets, active_mask, lse, ent = ctx.saved_tensors
        z = torch.zeros_like(lse)
        g = z if grad_logp is None else grad_logp.float().contiguous()
        gh = z if grad_entropy is None else grad_entropy.float().contiguous()
        dh, dw = linear_logp_entropy_bwd(hidden, weight, targets, active_mask, g, gh, lse, ent,
                                         ctx.temperature)
        return dh, dw, None, None, None


def linear_logp_entropy(hidden, weight, targets, active_mask=None, temperature=1.0):
    return LinearLogpEntropy.apply(hidden, weight, targets, active_mask, temperature)


class LinearKl(torch.autograd.Function):
    """(kl, kl_rev) = LinearKl.apply(hidden, weight, hidden_ref, weight_ref, active_mask, T, Tr);
    gradients flow to the policy head (hidden, weight) only."""

    @staticmethod
    def forward(ctx, hidden, weight, hidden_ref, weight_ref, active_mask, temperature,
                temperature_ref):
        kl, kl_rev, lse, lse_ref, _ = linear_kl_fwd(hidden, weight, hidden_ref, weight_ref,
                                                    active_mask, temperature, temperature_ref)
        ctx.save_for_backward(hidden, weight, hidden_ref, weight_ref, active_mask, lse, lse_ref,
                              kl)
        ctx.temperatures = (temperature, temperature_ref)
        return kl, kl_rev

    @staticmethod
    def backward(ctx, grad_kl, grad_kl_rev):
        hidden, weight, hidden_ref, weight_ref, active_mask, lse, lse_ref, kl = ctx.saved_tensors
        g = None if grad_kl is None else grad_kl.float().contiguous()
        gr = None if grad_kl_rev is None else grad_kl_rev.float().contiguous()
        if g is None and gr is None:
            return None, None, None, None, None, None, None
        dh, dw = linear_kl_bwd(hidden, weight, hidden_ref, weight_ref, active_mask, g, gr, lse,
                               lse_ref, kl, *ctx.temperatures)
        return dh, dw, None, None, None, None, None


def linear_kl(hidden, weight, hidden_ref, weight_ref, active_mask=None, temperature=1.0,
              temperature_ref=None):
    """Differentiable (kl, kl_rev) of the policy head against a fixed reference head."""
    temperature_ref = temperature if temperature_ref is None else temperature_ref
    return LinearKl.apply(hidden, weight, hidden_ref.detach(), weight_ref.detach(), active_mask,
                          temperature, temperature_ref)
