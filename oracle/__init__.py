"""CPU oracle for conv2d dgrad (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The CUDA library never links, loads or
calls it, and it imports nothing from the CUDA package.

The arithmetic lives in ``dgrad_oracle.c`` (plain double-precision loops
written from the definition; see that file's header for what each function
follows).  This module compiles it with gcc on first use into ``_build/`` and
exposes numpy-facing wrappers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "dgrad_oracle.c")
LIB_PATH = os.path.join(_HERE, "_build", "libdgrad_oracle.so")

_lock = threading.Lock()
_lib = None

_I = ctypes.c_int
_P = ctypes.c_void_p


def build_library(source: str = SOURCE, out_path: str = LIB_PATH) -> str:
    """Compile ``source`` (C) into the shared library ``out_path`` with gcc."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", source, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    shape = [_I] * 11
    lib.oracle_out_size.argtypes = [_I, _I, _I, _I]
    lib.oracle_out_size.restype = _I
    lib.oracle_dgrad_f64.argtypes = [_P, _P, _P] + shape + [_I, _I]
    lib.oracle_dgrad_f64.restype = _I
    lib.oracle_dgrad_points_f64.argtypes = [_P, _P, _P, ctypes.c_int64, _P] + shape + [_I]
    lib.oracle_dgrad_points_f64.restype = _I
    lib.oracle_conv2d_fwd_f64.argtypes = [_P, _P, _P] + shape + [_I]
    lib.oracle_conv2d_fwd_f64.restype = _I
    lib.oracle_shader_index_dgrad_f64.argtypes = [_P, _P, _P] + shape + [_I]
    lib.oracle_shader_index_dgrad_f64.restype = _I
    return lib


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library; ``path`` loads another copy."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            stale = (not os.path.exists(LIB_PATH)
                     or os.path.getmtime(LIB_PATH) < os.path.getmtime(SOURCE))
            if stale:
                build_library()
            _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def out_size(size: int, k: int, pad: int, stride: int, lib=None) -> int:
    """Output extent floor((size + 2*pad - k) / stride) + 1, or 0 if the kernel does not fit."""
    return (lib or load_library()).oracle_out_size(size, k, pad, stride)


def _shape_args(N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW):
    return [int(v) for v in (N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW)]


def dgrad(grad_out, weight, H: int, W: int, stride: int, padding_h: int, padding_w: int,
          nthreads: int = 0, lib=None, return_threads: bool = False):
    """grad_in [N,Ci,H,W] (float64) from grad_out [N,Co,OH,OW] and weight [Co,Ci,kH,kW]."""
    lib = lib or load_library()
    g, w = _f64(grad_out), _f64(weight)
    N, Co, OH, OW = g.shape
    Co2, Ci, kH, kW = w.shape
    assert Co == Co2, "grad_out and weight disagree on Co"
    out = np.empty((N, Ci, H, W), dtype=np.float64)
    args = _shape_args(N, Ci, H, W, Co, kH, kW, stride, padding_h, padding_w, OH, OW)
    t = lib.oracle_dgrad_f64(_ptr(g), _ptr(w), _ptr(out), *args, int(nthreads))
    if t < 0:
        raise ValueError("oracle rejected the shape")
    return (out, t) if return_threads else out


def dgrad_points(grad_out, weight, points, H: int, W: int, stride: int, padding_h: int,
                 padding_w: int, lib=None) -> np.ndarray:
    """grad_in at the given (n, ci, ih, iw) rows of ``points`` (int64 [P, 4])."""
    lib = lib or load_library()
    g, w = _f64(grad_out), _f64(weight)
    pts = np.ascontiguousarray(np.asarray(points, dtype=np.int64).reshape(-1, 4))
    N, Co, OH, OW = g.shape
    _, Ci, kH, kW = w.shape
    out = np.empty(pts.shape[0], dtype=np.float64)
    args = _shape_args(N, Ci, H, W, Co, kH, kW, stride, padding_h, padding_w, OH, OW)
    rc = lib.oracle_dgrad_points_f64(_ptr(g), _ptr(w), _ptr(pts), pts.shape[0], _ptr(out), *args)
    if rc != 0:
        raise ValueError(f"oracle rejected the points or shape (rc={rc})")
    return out


def conv2d_forward(x, weight, stride: int, padding_h: int, padding_w: int, lib=None) -> np.ndarray:
    """Forward conv out [N,Co,OH,OW] of x [N,Ci,H,W] with weight [Co,Ci,kH,kW]."""
    lib = lib or load_library()
    xx, w = _f64(x), _f64(weight)
    N, Ci, H, W = xx.shape
    Co, Ci2, kH, kW = w.shape
    assert Ci == Ci2
    OH = out_size(H, kH, padding_h, stride, lib)
    OW = out_size(W, kW, padding_w, stride, lib)
    out = np.empty((N, Co, OH, OW), dtype=np.float64)
    args = _shape_args(N, Ci, H, W, Co, kH, kW, stride, padding_h, padding_w, OH, OW)
    if lib.oracle_conv2d_fwd_f64(_ptr(xx), _ptr(w), _ptr(out), *args) != 0:
        raise ValueError("oracle rejected the shape")
    return out


def shader_index_dgrad(grad_out, weight, H: int, W: int, stride: int, padding_h: int,
                       padding_w: int, lib=None) -> np.ndarray:
    """The page's own index map restated (stride-1 shortcut); for documenting where it diverges."""
    lib = lib or load_library()
    g, w = _f64(grad_out), _f64(weight)
    N, Co, OH, OW = g.shape
    _, Ci, kH, kW = w.shape
    out = np.empty((N, Ci, H, W), dtype=np.float64)
    args = _shape_args(N, Ci, H, W, Co, kH, kW, stride, padding_h, padding_w, OH, OW)
    if lib.oracle_shader_index_dgrad_f64(_ptr(g), _ptr(w), _ptr(out), *args) != 0:
        raise ValueError("oracle rejected the shape")
    return out
