"""CPU oracle for the fused RMSNorm + matmul (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may import this module; the CUDA library never links, loads or calls it.  The
arithmetic lives in ``rmsnorm_matmul_oracle.c`` (plain double loops written
from the definition on the matmul_rms_norm.wgsl page; its header says what
each function follows), compiled with gcc on first use into ``_build/``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build_library

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "rmsnorm_matmul_oracle.c")
LIB_PATH = os.path.join(_HERE, "_build", "librmsnorm_oracle.so")

_lock = threading.Lock()
_lib = None
_I, _P, _D = ctypes.c_int, ctypes.c_void_p, ctypes.c_double


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.oracle_rms_rows_f64.argtypes = [_P, _P, _I, _I, _D]
    lib.oracle_rms_rows_f64.restype = _I
    lib.oracle_rms_normalize_f64.argtypes = [_P, _P, _P, _I, _I, _D]
    lib.oracle_rms_normalize_f64.restype = _I
    lib.oracle_rmsnorm_matmul_f64.argtypes = [_P, _P, _P, _P, _I, _I, _I, _D]
    lib.oracle_rmsnorm_matmul_f64.restype = _I
    return lib


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library; ``path`` loads another copy."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(SOURCE):
                build_library(SOURCE, LIB_PATH)
            _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def rms_rows(x, eps: float, lib=None) -> np.ndarray:
    """r[i] = 1 / sqrt(mean over t of X[i, t]^2 + eps) for X [M, K]."""
    lib = lib or load_library()
    xx = _f64(x)
    m, k = xx.shape
    r = np.empty(m, dtype=np.float64)
    if lib.oracle_rms_rows_f64(xx.ctypes.data, r.ctypes.data, m, k, float(eps)) != 0:
        raise ValueError("oracle rejected the shape")
    return r


def normalize(x, w_norm, eps: float, lib=None) -> np.ndarray:
    """The normalised operand A[i, t] = X[i, t] * r[i] * W_norm[t]."""
    lib = lib or load_library()
    xx, wn = _f64(x), _f64(w_norm)
    m, k = xx.shape
    assert wn.shape == (k,)
    a = np.empty((m, k), dtype=np.float64)
    if lib.oracle_rms_normalize_f64(xx.ctypes.data, wn.ctypes.data, a.ctypes.data, m, k, float(eps)) != 0:
        raise ValueError("oracle rejected the shape")
    return a


def rmsnorm_matmul(x, w_norm, w_proj, eps: float, lib=None) -> np.ndarray:
    """C [M, N] = RmsNorm(X, W_norm) x W_proj (float64)."""
    lib = lib or load_library()
    xx, wn, wp = _f64(x), _f64(w_norm), _f64(w_proj)
    m, k = xx.shape
    k2, n = wp.shape
    assert k == k2 and wn.shape == (k,)
    c = np.empty((m, n), dtype=np.float64)
    rc = lib.oracle_rmsnorm_matmul_f64(xx.ctypes.data, wn.ctypes.data, wp.ctypes.data, c.ctypes.data,
                                       m, n, k, float(eps))
    if rc != 0:
        raise ValueError("oracle rejected the shape")
    return c
