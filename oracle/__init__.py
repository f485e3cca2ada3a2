"""fp64 CPU oracle for the fused linear selected-token log-prob (test infrastructure).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product package never
imports this module, and this module never imports the product package: the
two share no code.  The arithmetic lives in ``rlk_oracle.c`` (plain loops in
IEEE double); this file only builds it, converts bf16 inputs to exact doubles
and marshals arrays through ctypes.

Every parity check in the suite pins the oracle first (closed forms,
high-precision brute force on tiny vocabularies, central finite differences,
hand-built audit vectors) before any GPU result is compared with it.

ctypes drops the GIL for the duration of each foreign call, so the helpers
``*_parallel`` below run independent rows of the (single-threaded) oracle on
several host threads; the arithmetic of each row is unchanged.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rlk_oracle.c")
_LIB = os.path.join(_HERE, "librlk_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u8p = ctypes.POINTER(ctypes.c_uint8)


class GrpoResult(ctypes.Structure):
    _fields_ = [
        ("active_count", ctypes.c_int64),
        ("clipped_count", ctypes.c_int64),
        ("outside_count", ctypes.c_int64),
        ("loss", ctypes.c_double),
        ("mean_ratio", ctypes.c_double),
    ]


class AuditExtResult(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("active_count", "argmax_index", "argmax_seq",
                                               "argmax_pos", "clip_count")] + \
               [(n, ctypes.c_double) for n in ("mean_dlogp", "mean_abs_dlogp", "mean_ratio",
                                                "approx_kl", "max_abs_dlogp", "p50_abs_dlogp",
                                                "p90_abs_dlogp", "p99_abs_dlogp", "clipfrac")]


class AuditResult(ctypes.Structure):
    _fields_ = [
        ("active_count", ctypes.c_int64),
        ("argmax_index", ctypes.c_int64),
        ("max_abs_dlogp", ctypes.c_double),
        ("mean_dlogp", ctypes.c_double),
        ("approx_kl", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile rlk_oracle.c with gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.rlk_oracle_linear_logp_fwd.restype = ctypes.c_int64
            lib.rlk_oracle_linear_logp_fwd.argtypes = [
                _dp, _dp, _i64p, _u8p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_double, _dp, _dp]
            for name in ("rlk_oracle_linear_logp_bwd_dh", "rlk_oracle_linear_logp_bwd_dw"):
                f = getattr(lib, name)
                f.restype = None
                f.argtypes = [_dp, _dp, _i64p, _u8p, _dp, _dp, ctypes.c_int64, ctypes.c_int64,
                              ctypes.c_int64, ctypes.c_double, ctypes.c_int64, ctypes.c_int64, _dp]
            lib.rlk_oracle_dlogp_audit.restype = None
            lib.rlk_oracle_dlogp_audit.argtypes = [_fp, _fp, _u8p, ctypes.c_int64,
                                                   ctypes.POINTER(AuditResult)]
            lib.rlk_oracle_grpo_clip.restype = None
            lib.rlk_oracle_grpo_clip.argtypes = [_dp, _dp, _dp, _u8p, ctypes.c_int64,
                                                 ctypes.c_double, ctypes.c_double,
                                                 ctypes.c_double, _dp, ctypes.POINTER(GrpoResult)]
            lib.rlk_oracle_logp_from_logits.restype = ctypes.c_int64
            lib.rlk_oracle_logp_from_logits.argtypes = [_dp, ctypes.c_int64, ctypes.c_int64,
                                                        _i64p, ctypes.c_int64, _i64p, _u8p,
                                                        ctypes.c_double, _dp, _dp]
            lib.rlk_oracle_linear_logp_entropy_fwd.restype = ctypes.c_int64
            lib.rlk_oracle_linear_logp_entropy_fwd.argtypes = [
                _dp, _dp, _i64p, _u8p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_double, _dp, _dp, _dp]
            for name in ("rlk_oracle_linear_logp_entropy_bwd_dh",
                         "rlk_oracle_linear_logp_entropy_bwd_dw"):
                f = getattr(lib, name)
                f.restype = None
                f.argtypes = [_dp, _dp, _i64p, _u8p, _dp, _dp, _dp, _dp, ctypes.c_int64,
                              ctypes.c_int64, ctypes.c_int64, ctypes.c_double, ctypes.c_int64,
                              ctypes.c_int64, _dp]
            lib.rlk_oracle_dlogp_audit_ext.restype = ctypes.c_int
            lib.rlk_oracle_dlogp_audit_ext.argtypes = [_fp, _fp, _u8p, ctypes.c_int64, _i64p,
                                                       ctypes.c_int64, ctypes.c_double,
                                                       ctypes.POINTER(AuditExtResult)]
            lib.rlk_oracle_linear_kl_fwd.restype = ctypes.c_int64
            lib.rlk_oracle_linear_kl_fwd.argtypes = [
                _dp, _dp, _dp, _dp, _u8p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_int64, ctypes.c_double, ctypes.c_double, _dp, _dp, _dp, _dp]
            for name in ("rlk_oracle_linear_kl_bwd_dh", "rlk_oracle_linear_kl_bwd_dw"):
                f = getattr(lib, name)
                f.restype = None
                f.argtypes = [_dp, _dp, _dp, _dp, _u8p, _dp, _dp, _dp, _dp, _dp, ctypes.c_int64,
                              ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
                              ctypes.c_double, ctypes.c_int64, ctypes.c_int64, _dp]
            lib.rlk_oracle_grpo_clip_grad.restype = ctypes.c_double
            lib.rlk_oracle_grpo_clip_grad.argtypes = [_dp, _dp, _dp, _u8p, ctypes.c_int64,
                                                      ctypes.c_double, _dp]
            _lib = lib
    return _lib


# ----------------------------------------------------------------------------- conversions

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact conversion of bf16 bit patterns (uint16 array or torch bf16 tensor) to float64."""
    if hasattr(bits, "view") and hasattr(bits, "dtype") and "bfloat16" in str(bits.dtype):
        bits = bits.contiguous().view(dtype=__import__("torch").int16).numpy().view(np.uint16)
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    flat_in = b.reshape(-1)
    flat_out = out.reshape(-1)
    step = 1 << 24
    for i in range(0, flat_in.size, step):
        seg = flat_in[i:i + step].astype(np.uint32) << np.uint32(16)
        flat_out[i:i + step] = seg.view(np.float32)
    return out


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _ptr(a, ctype):
    return a.ctypes.data_as(ctype) if a is not None else None


def _mask_arg(mask, n):
    if mask is None:
        return None
    m = _c(mask, np.uint8)
    assert m.shape == (n,)
    return m


# ----------------------------------------------------------------------------- forward / backward

def linear_logp_fwd(h, w, y, mask, temperature):
    """logp[N], lse[N] (float64) for h[N,H], W[V,H] given as exact float64 values."""
    lib = _load()
    h = _c(h, np.float64)
    w = _c(w, np.float64)
    n, hdim = h.shape
    vocab = w.shape[0]
    assert w.shape[1] == hdim
    y = _c(y, np.int64)
    m = _mask_arg(mask, n)
    logp = np.empty(n, np.float64)
    lse = np.empty(n, np.float64)
    bad = lib.rlk_oracle_linear_logp_fwd(_ptr(h, _dp), _ptr(w, _dp), _ptr(y, _i64p), _ptr(m, _u8p),
                                         n, hdim, vocab, float(temperature), _ptr(logp, _dp),
                                         _ptr(lse, _dp))
    if bad < 0:
        raise MemoryError("oracle forward: scratch allocation failed")
    return logp, lse


def linear_logp_fwd_parallel(h, w, y, mask, temperature, threads=None):
    """Same as linear_logp_fwd, rows split over host threads (each row computed alone)."""
    h = _c(h, np.float64)
    w = _c(w, np.float64)
    n = h.shape[0]
    y = _c(y, np.int64)
    m = _mask_arg(mask, n)
    threads = threads or max(1, len(os.sched_getaffinity(0)))
    bounds = np.linspace(0, n, min(threads, max(n, 1)) + 1).astype(np.int64)
    logp = np.empty(n, np.float64)
    lse = np.empty(n, np.float64)

    def work(i):
        a, b = int(bounds[i]), int(bounds[i + 1])
        if a == b:
            return
        lp, ls = linear_logp_fwd(h[a:b], w, y[a:b], None if m is None else m[a:b], temperature)
        logp[a:b] = lp
        lse[a:b] = ls

    with ThreadPoolExecutor(len(bounds) - 1) as ex:
        list(ex.map(work, range(len(bounds) - 1)))
    return logp, lse


def linear_logp_bwd_dh(h, w, y, mask, g, lse, temperature, row_begin=0, row_end=None):
    lib = _load()
    h = _c(h, np.float64)
    w = _c(w, np.float64)
    n, hdim = h.shape
    vocab = w.shape[0]
    row_end = n if row_end is None else row_end
    y = _c(y, np.int64)
    m = _mask_arg(mask, n)
    g = _c(g, np.float64)
    lse = _c(lse, np.float64)
    out = np.empty((row_end - row_begin, hdim), np.float64)
    lib.rlk_oracle_linear_logp_bwd_dh(_ptr(h, _dp), _ptr(w, _dp), _ptr(y, _i64p), _ptr(m, _u8p),
                                      _ptr(g, _dp), _ptr(lse, _dp), n, hdim, vocab,
                                      float(temperature), row_begin, row_end, _ptr(out, _dp))
    return out


def linear_logp_bwd_dw(h, w, y, mask, g, lse, temperature, v_begin=0, v_end=None):
    lib = _load()
    h = _c(h, np.float64)
    w = _c(w, np.float64)
    n, hdim = h.shape
    vocab = w.shape[0]
    v_end = vocab if v_end is None else v_end
    y = _c(y, np.int64)
    m = _mask_arg(mask, n)
    g = _c(g, np.float64)
    lse = _c(lse, np.float64)
    out = np.empty((v_end - v_begin, hdim), np.float64)
    lib.rlk_oracle_linear_logp_bwd_dw(_ptr(h, _dp), _ptr(w, _dp), _ptr(y, _i64p), _ptr(m, _u8p),
                                      _ptr(g, _dp), _ptr(lse, _dp), n, hdim, vocab,
                                      float(temperature), v_begin, v_end, _ptr(out, _dp))
    return out


def _split_parallel(total, fn, threads):
    threads = threads or max(1, len(os.sched_getaffinity(0)))
    parts = min(threads, max(total, 1))
    bounds = np.linspace(0, total, parts + 1).astype(np.int64)
    with ThreadPoolExecutor(parts) as ex:
        list(ex.map(lambda i: fn(int(bounds[i]), int(bounds[i + 1])), range(parts)))


def linear_logp_bwd_dh_parallel(h, w, y, mask, g, lse, temperature, threads=None):
    h = _c(h, np.float64)
    w = _c(w, np.float64)
    n, hdim = h.shape
    out = np.empty((n, hdim), np.float64)

    def fn(a, b):
        if a < b:
            out[a:b] = linear_logp_bwd_dh(h, w, y, mask, g, lse, temperature, a, b)

    _split_parallel(n, fn, threads)
    return out


def linear_logp_bwd_dw_parallel(h, w, y, mask, g, lse, temperature, v_begin, v_end, threads=None):
    h = _c(h, np.float64)
    w = _c(w, np.float64)
    out = np.empty((v_end - v_begin, h.shape[1]), np.float64)

    def fn(a, b):
        if a < b:
            out[a:b] = linear_logp_bwd_dw(h, w, y, mask, g, lse, temperature,
                                          v_begin + a, v_begin + b)

    _split_parallel(v_end - v_begin, fn, threads)
    return out


def linear_logp_bwd_dw_blocks(h, w, y, mask, g, lse, temperature, v_begin, v_end, consume,
                              rows_per_block=256, threads=None):
    """dW rows [v_begin, v_end) in blocks of rows_per_block, each handed to
    consume(v0, block) (called from worker threads) instead of being stored;
    the rows are computed exactly as by linear_logp_bwd_dw."""
    h = _c(h, np.float64)
    w = _c(w, np.float64)
    starts = list(range(v_begin, v_end, rows_per_block))
    threads = threads or max(1, len(os.sched_getaffinity(0)))

    def fn(v0):
        v1 = min(v_end, v0 + rows_per_block)
        consume(v0, linear_logp_bwd_dw(h, w, y, mask, g, lse, temperature, v0, v1))

    with ThreadPoolExecutor(min(threads, max(1, len(starts)))) as ex:
        list(ex.map(fn, starts))


# ----------------------------------------------------------------------------- audit / loss

def dlogp_audit(logp_new, logp_old, mask):
    lib = _load()
    a = _c(logp_new, np.float32)
    b = _c(logp_old, np.float32)
    n = a.shape[0]
    m = _mask_arg(mask, n)
    res = AuditResult()
    lib.rlk_oracle_dlogp_audit(_ptr(a, _fp), _ptr(b, _fp), _ptr(m, _u8p), n, ctypes.byref(res))
    return {
        "active_count": res.active_count,
        "argmax_index": res.argmax_index,
        "max_abs_dlogp": res.max_abs_dlogp,
        "mean_dlogp": res.mean_dlogp,
        "approx_kl": res.approx_kl,
    }


def grpo_clip_grad(logp, old, adv, mask, eps):
    """(loss, g[N]) of the GRPO clipped-ratio objective, token-mean over active tokens."""
    lib = _load()
    lp = _c(logp, np.float64)
    od = _c(old, np.float64)
    ad = _c(adv, np.float64)
    n = lp.shape[0]
    m = _mask_arg(mask, n)
    g = np.empty(n, np.float64)
    loss = lib.rlk_oracle_grpo_clip_grad(_ptr(lp, _dp), _ptr(od, _dp), _ptr(ad, _dp),
                                         _ptr(m, _u8p), n, float(eps), _ptr(g, _dp))
    return loss, g


def grpo_clip(logp, old, adv, mask, eps_low, eps_high, scale):
    """(g[N], result dict) of the clipped-ratio fragment with explicit range and scale."""
    lib = _load()
    lp = _c(logp, np.float64)
    od = _c(old, np.float64)
    ad = _c(adv, np.float64)
    n = lp.shape[0]
    m = _mask_arg(mask, n)
    g = np.empty(n, np.float64)
    res = GrpoResult()
    lib.rlk_oracle_grpo_clip(_ptr(lp, _dp), _ptr(od, _dp), _ptr(ad, _dp), _ptr(m, _u8p), n,
                             float(eps_low), float(eps_high), float(scale), _ptr(g, _dp),
                             ctypes.byref(res))
    return g, {f: getattr(res, f) for f, _ in GrpoResult._fields_}


def logp_from_logits(logits, y, mask, temperature, rows=None):
    """logp, lse (float64) of the selected rows of logits[N, V] (exact float64 values)."""
    lib = _load()
    z = _c(logits, np.float64)
    n, vocab = z.shape
    y = _c(y, np.int64)
    m = _mask_arg(mask, n)
    r = None if rows is None else _c(rows, np.int64)
    cnt = n if r is None else r.shape[0]
    logp = np.empty(cnt, np.float64)
    lse = np.empty(cnt, np.float64)
    lib.rlk_oracle_logp_from_logits(_ptr(z, _dp), vocab, vocab, _ptr(r, _i64p), cnt,
                                    _ptr(y, _i64p), _ptr(m, _u8p), float(temperature),
                                    _ptr(logp, _dp), _ptr(lse, _dp))
    return logp, lse


def linear_logp_entropy_fwd(h, w, y, mask, temperature):
    """logp[N], lse[N], entropy[N] (float64)."""
    lib = _load()
    h = _c(h, np.float64)
    w = _c(w, np.float64)
    n, hdim = h.shape
    y = _c(y, np.int64)
    m = _mask_arg(mask, n)
    logp, lse, ent = (np.empty(n, np.float64) for _ in range(3))
    if lib.rlk_oracle_linear_logp_entropy_fwd(_ptr(h, _dp), _ptr(w, _dp), _ptr(y, _i64p),
                                              _ptr(m, _u8p), n, hdim, w.shape[0],
                                              float(temperature), _ptr(logp, _dp),
                                              _ptr(lse, _dp), _ptr(ent, _dp)) < 0:
        raise MemoryError("oracle forward: scratch allocation failed")
    return logp, lse, ent


def linear_logp_entropy_fwd_parallel(h, w, y, mask, temperature, threads=None):
    h = _c(h, np.float64)
    w = _c(w, np.float64)
    n = h.shape[0]
    y = _c(y, np.int64)
    m = _mask_arg(mask, n)
    out = [np.empty(n, np.float64) for _ in range(3)]

    def fn(a, b):
        if a < b:
            r = linear_logp_entropy_fwd(h[a:b], w, y[a:b], None if m is None else m[a:b],
                                        temperature)
            for o, x in zip(out, r):
                o[a:b] = x

    _split_parallel(n, fn, threads)
    return tuple(out)


def _entropy_bwd(name, h, w, y, mask, g, gh, lse, ent, temperature, begin, end, rows):
    lib = _load()
    h = _c(h, np.float64)
    w = _c(w, np.float64)
    n, hdim = h.shape
    y = _c(y, np.int64)
    m = _mask_arg(mask, n)
    g, gh, lse, ent = (_c(x, np.float64) for x in (g, gh, lse, ent))
    out = np.empty((end - begin, hdim), np.float64)
    getattr(lib, name)(_ptr(h, _dp), _ptr(w, _dp), _ptr(y, _i64p), _ptr(m, _u8p), _ptr(g, _dp),
                       _ptr(gh, _dp), _ptr(lse, _dp), _ptr(ent, _dp), n, hdim, w.shape[0],
                       float(temperature), begin, end, _ptr(out, _dp))
    return out


def linear_logp_entropy_bwd_dh(h, w, y, mask, g, gh, lse, ent, temperature, row_begin=0,
                               row_end=None):
    row_end = np.asarray(h).shape[0] if row_end is None else row_end
    return _entropy_bwd("rlk_oracle_linear_logp_entropy_bwd_dh", h, w, y, mask, g, gh, lse, ent,
                        temperature, row_begin, row_end, True)


def linear_logp_entropy_bwd_dw(h, w, y, mask, g, gh, lse, ent, temperature, v_begin=0,
                               v_end=None):
    v_end = np.asarray(w).shape[0] if v_end is None else v_end
    return _entropy_bwd("rlk_oracle_linear_logp_entropy_bwd_dw", h, w, y, mask, g, gh, lse, ent,
                        temperature, v_begin, v_end, False)


def linear_logp_entropy_bwd_dh_parallel(h, w, y, mask, g, gh, lse, ent, temperature,
                                        threads=None):
    h = _c(h, np.float64)
    out = np.empty(h.shape, np.float64)

    def fn(a, b):
        if a < b:
            out[a:b] = linear_logp_entropy_bwd_dh(h, w, y, mask, g, gh, lse, ent, temperature,
                                                  a, b)

    _split_parallel(h.shape[0], fn, threads)
    return out


def linear_logp_entropy_bwd_dw_parallel(h, w, y, mask, g, gh, lse, ent, temperature,
                                        threads=None):
    w = _c(w, np.float64)
    out = np.empty(w.shape, np.float64)

    def fn(a, b):
        if a < b:
            out[a:b] = linear_logp_entropy_bwd_dw(h, w, y, mask, g, gh, lse, ent, temperature,
                                                  a, b)

    _split_parallel(w.shape[0], fn, threads)
    return out


def linear_kl_fwd(h, w, hr, wr, mask, temperature, temperature_ref):
    """Full-vocabulary KL of the policy head (h, W, T) against a reference head
    (hr, Wr, Tr): kl = KL(p || q), kl_rev = KL(q || p), lse, lse_ref (float64 [N])."""
    lib = _load()
    h, w, hr, wr = (_c(x, np.float64) for x in (h, w, hr, wr))
    n, hdim = h.shape
    m = _mask_arg(mask, n)
    out = [np.empty(n, np.float64) for _ in range(4)]
    if lib.rlk_oracle_linear_kl_fwd(_ptr(h, _dp), _ptr(w, _dp), _ptr(hr, _dp), _ptr(wr, _dp),
                                    _ptr(m, _u8p), n, hdim, hr.shape[1], w.shape[0],
                                    float(temperature), float(temperature_ref),
                                    *(_ptr(o, _dp) for o in out)) < 0:
        raise MemoryError("oracle KL forward: scratch allocation failed")
    return tuple(out)


def linear_kl_fwd_parallel(h, w, hr, wr, mask, temperature, temperature_ref, threads=None):
    h, w, hr, wr = (_c(x, np.float64) for x in (h, w, hr, wr))
    n = h.shape[0]
    m = _mask_arg(mask, n)
    out = [np.empty(n, np.float64) for _ in range(4)]

    def fn(a, b):
        if a < b:
            r = linear_kl_fwd(h[a:b], w, hr[a:b], wr, None if m is None else m[a:b],
                              temperature, temperature_ref)
            for o, x in zip(out, r):
                o[a:b] = x

    _split_parallel(n, fn, threads)
    return tuple(out)


def _kl_bwd(name, h, w, hr, wr, mask, g, gr, lse, lse_ref, kl, temperature, temperature_ref,
            begin, end, width):
    lib = _load()
    h, w, hr, wr = (_c(x, np.float64) for x in (h, w, hr, wr))
    n, hdim = h.shape
    m = _mask_arg(mask, n)
    g, gr, lse, lse_ref, kl = (_c(x, np.float64) for x in (g, gr, lse, lse_ref, kl))
    out = np.empty((end - begin, width), np.float64)
    getattr(lib, name)(_ptr(h, _dp), _ptr(w, _dp), _ptr(hr, _dp), _ptr(wr, _dp), _ptr(m, _u8p),
                       _ptr(g, _dp), _ptr(gr, _dp), _ptr(lse, _dp), _ptr(lse_ref, _dp),
                       _ptr(kl, _dp), n, hdim, hr.shape[1], w.shape[0], float(temperature),
                       float(temperature_ref), begin, end, _ptr(out, _dp))
    return out


def linear_kl_bwd_dh(h, w, hr, wr, mask, g, gr, lse, lse_ref, kl, temperature, temperature_ref,
                     row_begin=0, row_end=None):
    """Rows [row_begin, row_end) of dL/dh for L = sum g kl + sum gr kl_rev."""
    row_end = np.asarray(h).shape[0] if row_end is None else row_end
    return _kl_bwd("rlk_oracle_linear_kl_bwd_dh", h, w, hr, wr, mask, g, gr, lse, lse_ref, kl,
                   temperature, temperature_ref, row_begin, row_end, np.asarray(h).shape[1])


def linear_kl_bwd_dw(h, w, hr, wr, mask, g, gr, lse, lse_ref, kl, temperature, temperature_ref,
                     v_begin=0, v_end=None):
    """Rows [v_begin, v_end) of dL/dW for L = sum g kl + sum gr kl_rev."""
    v_end = np.asarray(w).shape[0] if v_end is None else v_end
    return _kl_bwd("rlk_oracle_linear_kl_bwd_dw", h, w, hr, wr, mask, g, gr, lse, lse_ref, kl,
                   temperature, temperature_ref, v_begin, v_end, np.asarray(h).shape[1])


def linear_kl_bwd_dh_parallel(h, w, hr, wr, mask, g, gr, lse, lse_ref, kl, temperature,
                              temperature_ref, threads=None):
    h = _c(h, np.float64)
    out = np.empty(h.shape, np.float64)

    def fn(a, b):
        if a < b:
            out[a:b] = linear_kl_bwd_dh(h, w, hr, wr, mask, g, gr, lse, lse_ref, kl, temperature,
                                        temperature_ref, a, b)

    _split_parallel(h.shape[0], fn, threads)
    return out


def linear_kl_bwd_dw_parallel(h, w, hr, wr, mask, g, gr, lse, lse_ref, kl, temperature,
                              temperature_ref, threads=None):
    w = _c(w, np.float64)
    out = np.empty((w.shape[0], np.asarray(h).shape[1]), np.float64)

    def fn(a, b):
        if a < b:
            out[a:b] = linear_kl_bwd_dw(h, w, hr, wr, mask, g, gr, lse, lse_ref, kl, temperature,
                                        temperature_ref, a, b)

    _split_parallel(w.shape[0], fn, threads)
    return out


def dlogp_audit_ext(logp_new, logp_old, mask, seq_offsets=None, eps=0.2):
    """The minimum diagnostics of the consistency contract (dict)."""
    lib = _load()
    a = _c(logp_new, np.float32)
    b = _c(logp_old, np.float32)
    n = a.shape[0]
    m = _mask_arg(mask, n)
    off = None if seq_offsets is None else _c(seq_offsets, np.int64)
    res = AuditExtResult()
    if lib.rlk_oracle_dlogp_audit_ext(_ptr(a, _fp), _ptr(b, _fp), _ptr(m, _u8p), n,
                                      _ptr(off, _i64p), 0 if off is None else off.shape[0] - 1,
                                      float(eps), ctypes.byref(res)) != 0:
        raise MemoryError("oracle audit: scratch allocation failed")
    return {f: getattr(res, f) for f, _ in AuditExtResult._fields_}
