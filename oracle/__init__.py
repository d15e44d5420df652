"""Float64 CPU oracle for the fused row reductions -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The product library never loads
it, and it imports nothing from the product package: the two share no code.

The arithmetic lives in ``oracle.c`` (plain C99, float64, one row at a time);
this module only compiles it with gcc, loads it with ctypes and marshals numpy
arrays.  Storage dtypes: float32 arrays are IEEE float32, uint16 arrays hold
bfloat16 bit patterns.  Every result is float64.

Definitions followed (page titles as published):
  * "Engineering a CUDA Machine Learning Framework from Scratch", sec. 3.1
    (three-pass softmax, online normaliser), sec. 3.2 (Welford LayerNorm),
    sec. 2.1 (loss gradient fused with the normalisation), sec. 2.2 (analytic
    backward);
  * "gpu-ml-learning" README, Module 3 (softmax, cross-entropy).
The online-softmax and Welford/Chan recurrences, whose equations were lost
from the pages, are restated from Milakov & Gimelshein (2018), Welford (1962)
and Chan, Golub & LeVeque (1979).  Attention (the pages' named extension of
the online softmax, "Engineering a CUDA Machine Learning Framework from
Scratch" sec. 6.4) is scaled dot-product attention as defined by Vaswani et
al. (2017), computed here by its plain three-pass definition per query row.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1

_dp = ctypes.POINTER(ctypes.c_double)
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-fno-fast-math", "-ffp-contract=off",
             "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_softmax.argtypes = [_vp, ctypes.c_int, _i64, _i64, _dp]
            lib.oracle_softmax.restype = None
            lib.oracle_xent.argtypes = [_vp, _vp, ctypes.c_int, _i64, _i64,
                                        ctypes.c_int32, _dp, _dp]
            lib.oracle_xent.restype = _i64
            lib.oracle_ln_fwd.argtypes = [_vp, _vp, _vp, ctypes.c_int, _i64, _i64,
                                          ctypes.c_double, _dp, _dp, _dp]
            lib.oracle_ln_fwd.restype = None
            lib.oracle_ln_bwd.argtypes = [_vp, _vp, _dp, _dp, _vp, ctypes.c_int,
                                          _i64, _i64, _dp, _dp, _dp, _dp, _dp]
            lib.oracle_ln_bwd.restype = None
            lib.oracle_softmax_bwd.argtypes = [_vp, _vp, ctypes.c_int, _i64, _i64, _dp]
            lib.oracle_softmax_bwd.restype = None
            lib.oracle_log_softmax.argtypes = [_vp, ctypes.c_int, _i64, _i64, _dp]
            lib.oracle_log_softmax.restype = None
            lib.oracle_log_softmax_bwd.argtypes = [_vp, _vp, ctypes.c_int, _i64, _i64, _dp]
            lib.oracle_log_softmax_bwd.restype = None
            lib.oracle_rms_fwd.argtypes = [_vp, _vp, ctypes.c_int, _i64, _i64, ctypes.c_double,
                                           _dp, _dp]
            lib.oracle_rms_fwd.restype = None
            lib.oracle_rms_bwd.argtypes = [_vp, _vp, _dp, _vp, ctypes.c_int, _i64, _i64, _dp,
                                           _dp, _dp]
            lib.oracle_rms_bwd.restype = None
            lib.oracle_online_softmax_stats.argtypes = [_dp, _i64, _dp, _dp]
            lib.oracle_online_softmax_stats.restype = None
            lib.oracle_online_merge.argtypes = [ctypes.c_double] * 4 + [_dp, _dp]
            lib.oracle_online_merge.restype = None
            lib.oracle_welford.argtypes = [_dp, _i64, _dp, _dp]
            lib.oracle_welford.restype = None
            lib.oracle_chan_merge.argtypes = [ctypes.c_double] * 6 + [_dp, _dp, _dp]
            lib.oracle_chan_merge.restype = None
            lib.oracle_attention.argtypes = [_vp, _vp, _vp, ctypes.c_int, _i64, _i64, _i64,
                                             ctypes.c_double, ctypes.c_int, _dp, _dp, _dp]
            lib.oracle_attention.restype = None
            _lib = lib
    return _lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle takes float32 or uint16 (bfloat16 bits), got {a.dtype}")


def _c(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_vp)


def _dptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def softmax(x: np.ndarray) -> np.ndarray:
    """Three-pass softmax of each row of a 2-D array; float64 result."""
    x = _c(x)
    rows, cols = x.shape
    y = np.empty((rows, cols), np.float64)
    _load().oracle_softmax(_ptr(x), _dtype_code(x), rows, cols, _dptr(y))
    return y


def xent(logits: np.ndarray, labels: np.ndarray, ignore_index: int = -100,
         want_dlogits: bool = True):
    """Per-row softmax cross-entropy and its gradient.

    Returns (loss[rows], dlogits[rows, cols] or None, bad_label_count)."""
    logits = _c(logits)
    labels = _c(labels.astype(np.int32, copy=False))
    rows, cols = logits.shape
    loss = np.empty(rows, np.float64)
    dl = np.empty((rows, cols), np.float64) if want_dlogits else None
    bad = _load().oracle_xent(_ptr(logits), _ptr(labels), _dtype_code(logits), rows,
                              cols, int(ignore_index), _dptr(loss), _dptr(dl))
    return loss, dl, int(bad)


def ln_fwd(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float,
           want_y: bool = True):
    """LayerNorm forward with two-pass moments.  Returns (y or None, mean, rstd)."""
    x, gamma, beta = _c(x), _c(gamma), _c(beta)
    code = _dtype_code(x)
    if _dtype_code(gamma) != code or _dtype_code(beta) != code:
        raise TypeError("x, gamma and beta must share one storage dtype")
    rows, cols = x.shape
    y = np.empty((rows, cols), np.float64) if want_y else None
    mean = np.empty(rows, np.float64)
    rstd = np.empty(rows, np.float64)
    _load().oracle_ln_fwd(_ptr(x), _ptr(gamma), _ptr(beta), code, rows, cols,
                          float(eps), _dptr(y), _dptr(mean), _dptr(rstd))
    return y, mean, rstd


def ln_bwd(dy: np.ndarray, x: np.ndarray, mean: np.ndarray, rstd: np.ndarray,
           gamma: np.ndarray, want_dx: bool = True):
    """LayerNorm backward from the saved statistics (float64 mean / rstd).

    Returns (dx or None, dgamma, dbeta, sum|dy*xhat| per column, sum|dy| per column)."""
    dy, x, gamma = _c(dy), _c(x), _c(gamma)
    mean = _c(np.asarray(mean, np.float64))
    rstd = _c(np.asarray(rstd, np.float64))
    code = _dtype_code(x)
    if _dtype_code(dy) != code or _dtype_code(gamma) != code:
        raise TypeError("dy, x and gamma must share one storage dtype")
    rows, cols = x.shape
    dx = np.empty((rows, cols), np.float64) if want_dx else None
    dg = np.empty(cols, np.float64)
    db = np.empty(cols, np.float64)
    dga = np.empty(cols, np.float64)
    dba = np.empty(cols, np.float64)
    _load().oracle_ln_bwd(_ptr(dy), _ptr(x), _dptr(mean), _dptr(rstd), _ptr(gamma),
                          code, rows, cols, _dptr(dx), _dptr(dg), _dptr(db),
                          _dptr(dga), _dptr(dba))
    return dx, dg, db, dga, dba


def softmax_bwd(y: np.ndarray, dy: np.ndarray) -> np.ndarray:
    """Softmax vector-Jacobian product dx = y * (dy - sum(y * dy)) per row."""
    y, dy = _c(y), _c(dy)
    code = _dtype_code(y)
    if _dtype_code(dy) != code:
        raise TypeError("y and dy must share one storage dtype")
    rows, cols = y.shape
    dx = np.empty((rows, cols), np.float64)
    _load().oracle_softmax_bwd(_ptr(y), _ptr(dy), code, rows, cols, _dptr(dx))
    return dx


def log_softmax(x: np.ndarray) -> np.ndarray:
    """Log-softmax of each row (x - max - ln sum exp(x - max)); masked rows 0."""
    x = _c(x)
    rows, cols = x.shape
    z = np.empty((rows, cols), np.float64)
    _load().oracle_log_softmax(_ptr(x), _dtype_code(x), rows, cols, _dptr(z))
    return z


def log_softmax_bwd(z: np.ndarray, dz: np.ndarray) -> np.ndarray:
    """Log-softmax vector-Jacobian product dx = dz - exp(z) * sum(dz) per row."""
    z, dz = _c(z), _c(dz)
    code = _dtype_code(z)
    if _dtype_code(dz) != code:
        raise TypeError("z and dz must share one storage dtype")
    rows, cols = z.shape
    dx = np.empty((rows, cols), np.float64)
    _load().oracle_log_softmax_bwd(_ptr(z), _ptr(dz), code, rows, cols, _dptr(dx))
    return dx


def rms_fwd(x: np.ndarray, gamma: np.ndarray, eps: float, want_y: bool = True):
    """RMSNorm forward.  Returns (y or None, rstd)."""
    x, gamma = _c(x), _c(gamma)
    code = _dtype_code(x)
    if _dtype_code(gamma) != code:
        raise TypeError("x and gamma must share one storage dtype")
    rows, cols = x.shape
    y = np.empty((rows, cols), np.float64) if want_y else None
    rstd = np.empty(rows, np.float64)
    _load().oracle_rms_fwd(_ptr(x), _ptr(gamma), code, rows, cols, float(eps), _dptr(y),
                           _dptr(rstd))
    return y, rstd


def rms_bwd(dy: np.ndarray, x: np.ndarray, rstd: np.ndarray, gamma: np.ndarray,
            want_dx: bool = True):
    """RMSNorm backward from the saved rstd (float64).

    Returns (dx or None, dgamma, sum|dy*xhat| per column)."""
    dy, x, gamma = _c(dy), _c(x), _c(gamma)
    rstd = _c(np.asarray(rstd, np.float64))
    code = _dtype_code(x)
    if _dtype_code(dy) != code or _dtype_code(gamma) != code:
        raise TypeError("dy, x and gamma must share one storage dtype")
    rows, cols = x.shape
    dx = np.empty((rows, cols), np.float64) if want_dx else None
    dg = np.empty(cols, np.float64)
    dga = np.empty(cols, np.float64)
    _load().oracle_rms_bwd(_ptr(dy), _ptr(x), _dptr(rstd), _ptr(gamma), code, rows, cols,
                           _dptr(dx), _dptr(dg), _dptr(dga))
    return dx, dg, dga


# -- self-check helpers: the recurrences the GPU path uses ----------------------

def online_softmax_stats(x: np.ndarray):
    """(m, d) of the one-pass online normaliser over a float64 vector."""
    x = _c(np.asarray(x, np.float64))
    m, d = ctypes.c_double(), ctypes.c_double()
    _load().oracle_online_softmax_stats(_dptr(x), x.size, ctypes.byref(m), ctypes.byref(d))
    return m.value, d.value


def online_merge(ma, da, mb, db):
    m, d = ctypes.c_double(), ctypes.c_double()
    _load().oracle_online_merge(ma, da, mb, db, ctypes.byref(m), ctypes.byref(d))
    return m.value, d.value


def welford(x: np.ndarray):
    """(mean, M2) of Welford's one-pass update over a float64 vector."""
    x = _c(np.asarray(x, np.float64))
    mean, m2 = ctypes.c_double(), ctypes.c_double()
    _load().oracle_welford(_dptr(x), x.size, ctypes.byref(mean), ctypes.byref(m2))
    return mean.value, m2.value


def chan_merge(na, mean_a, m2a, nb, mean_b, m2b):
    n, mean, m2 = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    _load().oracle_chan_merge(na, mean_a, m2a, nb, mean_b, m2b, ctypes.byref(n),
                              ctypes.byref(mean), ctypes.byref(m2))
    return n.value, mean.value, m2.value


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, causal: bool = True):
    """Scaled dot-product attention of [bh, s, d] arrays (float32 or bfloat16
    bits), causal or not; returns (o [bh, s, d], lse [bh, s]) in float64."""
    q, k, v = _c(q), _c(k), _c(v)
    if not (q.shape == k.shape == v.shape and q.ndim == 3):
        raise ValueError("q, k, v must share one [bh, s, d] shape")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one storage dtype")
    bh, s, d = q.shape
    o = np.empty((bh, s, d), np.float64)
    lse = np.empty((bh, s), np.float64)
    scratch = np.empty(max(1, s), np.float64)
    _load().oracle_attention(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), bh, s, d,
                             float(scale), 1 if causal else 0, _dptr(o), _dptr(lse),
                             _dptr(scratch))
    return o, lse
