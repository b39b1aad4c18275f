"""CPU oracle for the attention gradient with respect to V (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may import this module; the CUDA library never links, loads or calls it.  The
arithmetic lives in ``mha_grad_v_oracle.c`` (plain double loops written from
the mha_grad_v.wgsl page; its header states the definition), compiled with gcc
on first use into ``_build/``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build_library

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "mha_grad_v_oracle.c")
LIB_PATH = os.path.join(_HERE, "_build", "libmha_oracle.so")

_lock = threading.Lock()
_lib = None
_I, _P = ctypes.c_int, ctypes.c_void_p


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.oracle_mha_grad_v_f64.argtypes = [_P, _P, _P, _P, _P] + [_I] * 6
    lib.oracle_mha_grad_v_f64.restype = _I
    lib.oracle_mha_grad_v_rows_f64.argtypes = [_P, _P, _P, _P, _P] + [_I] * 8
    lib.oracle_mha_grad_v_rows_f64.restype = _I
    lib.oracle_mha_forward_lse_f64.argtypes = [_P, _P, _P] + [_I] * 6
    lib.oracle_mha_forward_lse_f64.restype = _I
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


def kv_len(q_seq: int, kv_seq: int) -> int:
    """Key/value positions: q_seq when kv_seq == 0 (causal), else kv_seq."""
    return q_seq if kv_seq == 0 else kv_seq


def forward_lse(q, k, kv_seq: int, window: int, lib=None) -> np.ndarray:
    """LSE [q_seq, num_heads, 2] = (max score, log sum exp(score - max)) over the
    keys each query attends; q [q_seq, H, d], k [kv, KVH, d]."""
    lib = lib or load_library()
    qq, kk = _f64(q), _f64(k)
    q_seq, nh, hd = qq.shape
    kv, nkv, hd2 = kk.shape
    assert hd == hd2 and kv == kv_len(q_seq, kv_seq)
    out = np.empty((q_seq, nh, 2), dtype=np.float64)
    if lib.oracle_mha_forward_lse_f64(qq.ctypes.data, kk.ctypes.data, out.ctypes.data, q_seq, kv_seq, nh, nkv,
                                      hd, window) != 0:
        raise ValueError("oracle rejected the shape")
    return out


def grad_v(q, k, d_out, lse, kv_seq: int, window: int, lib=None) -> np.ndarray:
    """dV [kv, KVH, d] of the page's definition (float64)."""
    lib = lib or load_library()
    qq, kk, go, ls = _f64(q), _f64(k), _f64(d_out), _f64(lse)
    q_seq, nh, hd = qq.shape
    kv, nkv, _ = kk.shape
    assert go.shape == qq.shape and ls.shape == (q_seq, nh, 2) and kv == kv_len(q_seq, kv_seq)
    dv = np.empty((kv, nkv, hd), dtype=np.float64)
    rc = lib.oracle_mha_grad_v_f64(qq.ctypes.data, kk.ctypes.data, go.ctypes.data, ls.ctypes.data, dv.ctypes.data,
                                   q_seq, kv_seq, nh, nkv, hd, window)
    if rc != 0:
        raise ValueError("oracle rejected the shape")
    return dv


def grad_v_rows(q, k, d_out, lse, kv_seq: int, window: int, t_begin: int, t_end: int, lib=None) -> np.ndarray:
    """Rows t_begin .. t_end - 1 of dV (float64), for checks at sizes where every row costs too much."""
    lib = lib or load_library()
    qq, kk, go, ls = _f64(q), _f64(k), _f64(d_out), _f64(lse)
    q_seq, nh, hd = qq.shape
    kv, nkv, _ = kk.shape
    assert go.shape == qq.shape and ls.shape == (q_seq, nh, 2) and kv == kv_len(q_seq, kv_seq)
    dv = np.empty((t_end - t_begin, nkv, hd), dtype=np.float64)
    rc = lib.oracle_mha_grad_v_rows_f64(qq.ctypes.data, kk.ctypes.data, go.ctypes.data, ls.ctypes.data,
                                        dv.ctypes.data, q_seq, kv_seq, nh, nkv, hd, window, t_begin, t_end)
    if rc != 0:
        raise ValueError("oracle rejected the shape or range")
    return dv
