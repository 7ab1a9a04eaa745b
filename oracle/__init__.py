"""ctypes front end of the plain C oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: the test-suite, the package smoke check and the
benchmark's CPU-baseline leg use it.  The product path never imports it.

Every function takes numpy arrays (or torch CPU tensors, converted here) and
returns numpy arrays.  bf16 logits travel as their raw 16-bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_NONFINITE = -4
F32, BF16 = 0, 1
MAX_DRAFT = 32

CFLAGS = ["-O2", "-std=c11", "-Wall", "-Wextra", "-shared", "-fPIC",
          "-ffp-contract=off", "-fexcess-precision=standard"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, seconds)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"], check=True)
        os.replace(tmp, LIB)
    return LIB


_lib = None
_lock = threading.Lock()

_p = ctypes.c_void_p
_i32, _i64, _f32, _f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double


def load(path: str | None = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        lib = ctypes.CDLL(path or build())
        lib.oracle_softmax_stats.argtypes = [_p, ctypes.c_int, _i64, _i64, _f64, _p, _p]
        lib.oracle_softmax_row.argtypes = [_p, ctypes.c_int, _i64, _i64, _f64, _p]
        lib.oracle_argmax_row.argtypes = [_p, ctypes.c_int, _i64, _i64, _p]
        lib.oracle_inverse_cdf.argtypes = [_p, _i64, _f64, _p, _p]
        lib.oracle_inverse_cdf.restype = _i64
        lib.oracle_verify_greedy.argtypes = [_p, ctypes.c_int, _p, _p, _i32, _i64, _i32, _p, _p]
        lib.oracle_verify_sample.argtypes = [_p, _p, ctypes.c_int, _p, _p, _i32, _i64, _i32,
                                             _f64, _p, _p, _p, _p, _p, _p, _p, _p]
        lib.oracle_final_weights.argtypes = [_p, _p, ctypes.c_int, _i64, _f64, _i64, _i64,
                                             _p, _p]
        lib.oracle_final_cdf.argtypes = [_p, _p, ctypes.c_int, _p, _i32, _i64, _i32, _f64,
                                         _i32, _p]
        lib.oracle_dcut_allocate.argtypes = [_p, _p, _i32, _i32, _i32, _f32, _p, _p, _p]
        lib.oracle_dcut_cost.argtypes = [_i32]
        lib.oracle_dcut_cost.restype = _f64
        lib.oracle_dcut_schedule_cost.argtypes = [_p, _p, _i32, _i32, _f64, _p, _p, _p]
        lib.oracle_draft_confidence.argtypes = [_p, ctypes.c_int, _p, _p, _i32, _i32, _i64, _f64,
                                                _p]
        lib.oracle_draft_sample.argtypes = [_p, ctypes.c_int, _p, _i32, _i32, _i64, _f64, _p, _p,
                                            _p]
        lib.oracle_acceptance_stats.argtypes = [_p, _p, _i32, _i32, _p, _p, _p]
        if path is None:
            _lib = lib
        return lib


# ---------------------------------------------------------------------------
# marshalling
# ---------------------------------------------------------------------------


def _np(x, dtype=None):
    """numpy view of x (torch CPU tensor or array), C-contiguous."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu()
            if x.dtype == torch.bfloat16:
                x = x.view(torch.int16).numpy().view(np.uint16)
            else:
                x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.asarray(x)
    if dtype is not None:
        x = x.astype(dtype, copy=False)
    return np.ascontiguousarray(x)


def _logits(x):
    """(array, dtype code) for float32 or bf16 (uint16 bit patterns) logits."""
    a = _np(x)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    if a.dtype == np.float64:
        raise TypeError("logits must be float32 or bf16; fp64 inputs are not a path dtype")
    raise TypeError(f"unsupported logits dtype {a.dtype}")


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


# ---------------------------------------------------------------------------
# row primitives
# ---------------------------------------------------------------------------


def softmax_stats(logits, row: int, T: float, lib=None):
    a, dt = _logits(logits)
    V = a.shape[-1]
    m, s = _f64(), _f64()
    st = (lib or load()).oracle_softmax_stats(_ptr(a), dt, row, V, T, ctypes.byref(m),
                                              ctypes.byref(s))
    return st, m.value, s.value


def softmax_row(logits, row: int, T: float, lib=None):
    a, dt = _logits(logits)
    V = a.shape[-1]
    out = np.zeros(V, np.float64)
    st = (lib or load()).oracle_softmax_row(_ptr(a), dt, row, V, T, _ptr(out))
    return st, out


def argmax_row(logits, row: int, lib=None):
    a, dt = _logits(logits)
    out = _i32(-7)
    st = (lib or load()).oracle_argmax_row(_ptr(a), dt, row, a.shape[-1], ctypes.byref(out))
    return st, out.value


def inverse_cdf(w, u: float, lib=None):
    w = _np(w, np.float64)
    uS, S = _f64(), _f64()
    v = (lib or load()).oracle_inverse_cdf(_ptr(w), w.size, u, ctypes.byref(uS),
                                           ctypes.byref(S))
    return v, uS.value, S.value


def final_weights(target, draft, trow: int, drow: int, T: float, lib=None):
    t, dt = _logits(target)
    d, dt2 = _logits(draft) if draft is not None else (t, dt)
    V = t.shape[-1]
    out = np.zeros(V, np.float64)
    fb = _i32(0)
    st = (lib or load()).oracle_final_weights(_ptr(t), _ptr(d), dt, V, T, trow, drow,
                                              _ptr(out), ctypes.byref(fb))
    return st, out, fb.value


# ---------------------------------------------------------------------------
# verification
# ---------------------------------------------------------------------------


class VerifyResult(dict):
    """tokens, accept_len, status, and (sampling) p, q, ratio, final."""

    def __getattr__(self, k):
        try:
            return self[k]
        except KeyError as e:  # pragma: no cover
            raise AttributeError(k) from e


def verify_greedy(target, draft_tokens, cu_draft, draft_stride: int = 0, lib=None):
    t, dt = _logits(target)
    tok = _np(draft_tokens, np.int32)
    cu = _np(cu_draft, np.int32)
    B = cu.size - 1
    V = t.shape[-1]
    rows = int(cu[-1]) + B if B > 0 else 0
    out_tokens = np.full(max(rows, 1), -7, np.int32)
    out_len = np.full(max(B, 1), -7, np.int32)
    st = (lib or load()).oracle_verify_greedy(_ptr(t), dt, _ptr(tok), _ptr(cu), B, V,
                                              draft_stride, _ptr(out_tokens), _ptr(out_len))
    return VerifyResult(status=st, tokens=out_tokens[:rows], accept_len=out_len[:B])


def verify_sample(target, draft, draft_tokens, cu_draft, temperature: float, u_accept,
                  u_final, draft_stride: int = 0, lib=None):
    t, dt = _logits(target)
    if draft is not None and _np(draft).shape[0] > 0:
        d, dt2 = _logits(draft)
        if dt2 != dt:
            raise TypeError("target and draft logits must share a dtype")
    else:
        d = t
    tok = _np(draft_tokens, np.int32)
    cu = _np(cu_draft, np.int32)
    ua = _np(u_accept, np.float32)
    uf = _np(u_final, np.float32)
    B = cu.size - 1
    V = t.shape[-1]
    rows = int(cu[-1]) + B if B > 0 else 0
    nd = max(tok.size, 1)
    out_tokens = np.full(max(rows, 1), -7, np.int32)
    out_len = np.full(max(B, 1), -7, np.int32)
    out_p = np.full(nd, np.nan, np.float32)
    out_q = np.full(nd, np.nan, np.float32)
    ratio = np.full(nd, np.nan, np.float64)
    final = np.full((max(B, 1), 4), np.nan, np.float64)
    st = (lib or load()).oracle_verify_sample(
        _ptr(t), _ptr(d), dt, _ptr(tok), _ptr(cu), B, V, draft_stride, float(temperature),
        _ptr(ua), _ptr(uf), _ptr(out_tokens), _ptr(out_len), _ptr(out_p), _ptr(out_q),
        _ptr(ratio), _ptr(final))
    return VerifyResult(status=st, tokens=out_tokens[:rows], accept_len=out_len[:B],
                        p=out_p[:tok.size], q=out_q[:tok.size], ratio=ratio[:tok.size],
                        final=final[:B])


def final_cdf(target, draft, cu_draft, i: int, a: int, temperature: float,
              draft_stride: int = 0, lib=None):
    t, dt = _logits(target)
    d = _logits(draft)[0] if draft is not None and _np(draft).shape[0] > 0 else t
    cu = _np(cu_draft, np.int32)
    V = t.shape[-1]
    out = np.zeros(V, np.float64)
    st = (lib or load()).oracle_final_cdf(_ptr(t), _ptr(d), dt, _ptr(cu), i, V, draft_stride,
                                          float(temperature), a, _ptr(out))
    return st, out


def dcut_allocate(conf, kmax, budget: int, min_gain: float = 0.0, lib=None):
    c = _np(conf, np.float32)
    km = _np(kmax, np.int32)
    B = km.size
    Kmax = c.shape[1] if c.ndim == 2 else (c.size // B if B else 0)
    depth = np.full(max(B, 1), -7, np.int32)
    cu = np.full(B + 1, -7, np.int32)
    exp_len = np.full(max(B, 1), np.nan, np.float64)
    st = (lib or load()).oracle_dcut_allocate(_ptr(c), _ptr(km), B, Kmax, budget,
                                              float(min_gain), _ptr(depth), _ptr(cu),
                                              _ptr(exp_len))
    return VerifyResult(status=st, depth=depth[:B], cu=cu, expected=exp_len[:B])


def dcut_cost(d: int, lib=None) -> float:
    return float((lib or load()).oracle_dcut_cost(int(d)))


def dcut_schedule_cost(conf, kmax, max_cost: float, lib=None):
    """The cost-unit D-cut variant: per-request best depth by benefit, then
    greedy admission under max_cost (latency-cost units)."""
    c = _np(conf, np.float32)
    km = _np(kmax, np.int32)
    B = km.size
    Kmax = c.shape[1] if c.ndim == 2 else (c.size // B if B else 0)
    depth = np.full(max(B, 1), -7, np.int32)
    cu = np.full(B + 1, -7, np.int32)
    benefit = np.full(max(B, 1), np.nan, np.float64)
    st = (lib or load()).oracle_dcut_schedule_cost(_ptr(c), _ptr(km), B, Kmax, float(max_cost),
                                                   _ptr(depth), _ptr(cu), _ptr(benefit))
    return VerifyResult(status=st, depth=depth[:B], cu=cu, benefit=benefit[:B])


def draft_confidence(draft, tokens, kmax, temperature: float, lib=None):
    """q_{i,j}(x_{i,j}) for padded draft rows [B*Kmax, V]; 0 past kmax[i]."""
    d, dt = _logits(draft)
    tok = _np(tokens, np.int32)
    km = _np(kmax, np.int32)
    B = km.size
    Kmax = tok.size // B if B else 0
    V = d.shape[-1]
    out = np.full(max(B * Kmax, 1), -7.0, np.float32)
    st = (lib or load()).oracle_draft_confidence(_ptr(d), dt, _ptr(tok), _ptr(km), B, Kmax, V,
                                                 float(temperature), _ptr(out))
    return st, out[:B * Kmax].reshape(B, Kmax) if B else out[:0]


def draft_sample(draft, kmax, Kmax: int, temperature: float, u, lib=None):
    """Drafted tokens x ~ q (inverse CDF at u) for padded rows; -1 past kmax."""
    d, dt = _logits(draft)
    km = _np(kmax, np.int32)
    uu = _np(u, np.float32)
    B = km.size
    V = d.shape[-1]
    tok = np.full(max(B * Kmax, 1), -7, np.int32)
    conf = np.full(max(B * Kmax, 1), -7.0, np.float32)
    st = (lib or load()).oracle_draft_sample(_ptr(d), dt, _ptr(km), B, Kmax, V,
                                             float(temperature), _ptr(uu), _ptr(tok), _ptr(conf))
    return st, tok[:B * Kmax], conf[:B * Kmax]


def acceptance_stats(accept_len, cu_draft, Kmax: int, lib=None):
    a = _np(accept_len, np.int32)
    cu = _np(cu_draft, np.int32)
    B = a.size
    reached = np.full(max(Kmax, 1), -7, np.int32)
    accepted = np.full(max(Kmax, 1), -7, np.int32)
    mean = _f64(-1.0)
    st = (lib or load()).oracle_acceptance_stats(_ptr(a), _ptr(cu), B, Kmax, _ptr(reached),
                                                 _ptr(accepted), ctypes.byref(mean))
    return st, reached[:Kmax], accepted[:Kmax], mean.value
