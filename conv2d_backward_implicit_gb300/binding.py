"""ctypes binding for the C ABI in include/conv2d_grad_input.h, include/rmsnorm_matmul.h
and include/mha_grad_v.h (argument marshalling only).

Every function here has the name of the C entry point it calls, accepts torch
tensors (or raw integer addresses) for the buffers, and raises
:class:`DgradError` when the C call returns a non-zero status.  No part of the
computation runs in Python, and there is no fallback: if the library has not
been built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build_ext

DGRAD_F32, DGRAD_BF16, DGRAD_F16 = 0, 1, 2
DGRAD_KERNEL_AUTO, DGRAD_KERNEL_TC, DGRAD_KERNEL_SIMT, DGRAD_KERNEL_TC_POSM = 0, 1, 2, 3
DGRAD_DEBUG_SKIP_ARRIVE = 1
STATUS = {
    0: "DGRAD_OK", 1: "DGRAD_ERR_INVALID_ARG", 2: "DGRAD_ERR_SHAPE", 3: "DGRAD_ERR_ALIGNMENT",
    4: "DGRAD_ERR_UNSUPPORTED", 5: "DGRAD_ERR_CUDA", 6: "DGRAD_ERR_TIMEOUT",
    7: "DGRAD_ERR_WORKSPACE",
}
DTYPE_CODE = {"f32": DGRAD_F32, "bf16": DGRAD_BF16, "f16": DGRAD_F16}

PARAM_FIELDS = ("batch", "in_channels", "in_h", "in_w", "out_channels", "kernel_h", "kernel_w",
                "stride", "padding_h", "out_h", "out_w", "padding_w")


class Params(ctypes.Structure):
    """conv2d_grad_input_params: twelve uint32 fields in the header's order."""
    _fields_ = [(name, ctypes.c_uint32) for name in PARAM_FIELDS]

    def as_dict(self):
        return {k: int(getattr(self, k)) for k in PARAM_FIELDS}


class RmsParams(ctypes.Structure):
    """rmsnorm_matmul_params: m, n, k (uint32) and eps (float)."""
    _fields_ = [("m", ctypes.c_uint32), ("n", ctypes.c_uint32), ("k", ctypes.c_uint32),
                ("eps", ctypes.c_float)]


MHA_FIELDS = ("q_seq", "kv_seq", "num_heads", "num_kv_heads", "head_dim", "window_size")


class MhaParams(ctypes.Structure):
    """mha_grad_v_params: six uint32 fields in the header's order."""
    _fields_ = [(name, ctypes.c_uint32) for name in MHA_FIELDS]


class DgradError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


def params_from_shapes(grad_out_shape, weight_shape, in_h: int, in_w: int, stride: int,
                       padding_h: int, padding_w: int) -> Params:
    """Fill Params from tensor shapes: grad_out [N,Co,OH,OW], weight [Co,Ci,kH,kW]."""
    N, Co, OH, OW = (int(v) for v in grad_out_shape)
    Co2, Ci, kH, kW = (int(v) for v in weight_shape)
    if Co != Co2:
        raise ValueError("grad_out and weight disagree on out_channels")
    return Params(N, Ci, in_h, in_w, Co, kH, kW, stride, padding_h, OH, OW, padding_w)


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return build_ext.LIB_PATH


def library() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is missing: build it with __graft_entry__.build() "
                    "(or python -m conv2d_backward_implicit_gb300.build_ext); there is no fallback")
            lib = ctypes.CDLL(path)
            P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            PP = ctypes.POINTER(Params)
            lib.conv2d_grad_input.argtypes = [P, P, P, PP, I, P]
            lib.conv2d_grad_input.restype = I
            lib.conv2d_grad_input_workspace_size.argtypes = [PP, I]
            lib.conv2d_grad_input_workspace_size.restype = S
            lib.conv2d_grad_input_pack_weight.argtypes = [P, P, S, PP, I, P]
            lib.conv2d_grad_input_pack_weight.restype = I
            lib.conv2d_grad_input_prepacked.argtypes = [P, P, P, PP, I, P]
            lib.conv2d_grad_input_prepacked.restype = I
            lib.conv2d_grad_input_check_errors.argtypes = [P]
            lib.conv2d_grad_input_check_errors.restype = I
            lib.conv2d_grad_input_status_string.argtypes = [I]
            lib.conv2d_grad_input_status_string.restype = ctypes.c_char_p
            lib.conv2d_grad_input_select_kernel.argtypes = [PP, I]
            lib.conv2d_grad_input_select_kernel.restype = I
            lib.conv2d_grad_input_set_kernel.argtypes = [I]
            lib.conv2d_grad_input_set_kernel.restype = I
            lib.conv2d_grad_input_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            lib.conv2d_grad_input_set_wait_limit_ns.restype = ctypes.c_uint64
            lib.conv2d_grad_input_set_debug.argtypes = [I]
            lib.conv2d_grad_input_set_debug.restype = I
            lib.conv2d_grad_input_noalloc.argtypes = [P, P, P, PP, I, P]
            lib.conv2d_grad_input_noalloc.restype = I
            lib.conv2d_forward.argtypes = [P, P, P, PP, I, P]
            lib.conv2d_forward.restype = I
            RP = ctypes.POINTER(RmsParams)
            lib.rmsnorm_matmul.argtypes = [P, P, P, P, RP, I, P]
            lib.rmsnorm_matmul.restype = I
            lib.rmsnorm_matmul_select_kernel.argtypes = [P, P, P, P, RP, I]
            lib.rmsnorm_matmul_select_kernel.restype = I
            lib.rmsnorm_matmul_set_kernel.argtypes = [I]
            lib.rmsnorm_matmul_set_kernel.restype = I
            lib.rmsnorm_matmul_check_errors.argtypes = [P]
            lib.rmsnorm_matmul_check_errors.restype = I
            MP = ctypes.POINTER(MhaParams)
            lib.mha_grad_v.argtypes = [P, P, P, P, P, MP, I, P]
            lib.mha_grad_v.restype = I
            lib.mha_grad_v_select_kernel.argtypes = [P, P, P, P, P, MP, I]
            lib.mha_grad_v_select_kernel.restype = I
            lib.mha_grad_v_set_kernel.argtypes = [I]
            lib.mha_grad_v_set_kernel.restype = I
            lib.mha_grad_v_check_errors.argtypes = [P]
            lib.mha_grad_v_check_errors.restype = I
            _lib = lib
    return _lib


_TORCH_DTYPE_NAME = {DGRAD_F32: "float32", DGRAD_BF16: "bfloat16", DGRAD_F16: "float16"}
_ESIZE = {DGRAD_F32: 4, DGRAD_BF16: 2, DGRAD_F16: 2}


def _current_device() -> int:
    import torch
    return int(torch.cuda.current_device())


def _addr(x, name: str = "buffer", dtype: str | None = None, numel: int | None = None,
          min_bytes: int | None = None) -> int | None:
    """Device address of a buffer argument.  Integers pass through unchecked;
    a tensor must live on the current CUDA device (the library launches there),
    be contiguous (the C ABI reads dense NCHW / [Co,Ci,kH,kW] memory), have the
    element type ``dtype`` and exactly ``numel`` elements when those are given,
    and hold at least ``min_bytes`` bytes -- all checked here, on the host,
    before the library is called, so a tensor smaller than the Params describe
    never reaches a kernel."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    dev = getattr(x, "device", None)
    if dev is not None and getattr(dev, "type", "cuda") != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got one on {dev})")
    index = getattr(dev, "index", None) if dev is not None else None
    if index is not None and int(index) != _current_device():
        raise ValueError(f"{name} is on cuda:{index} but the current device is "
                         f"cuda:{_current_device()}: the library launches on the current device")
    if hasattr(x, "is_contiguous") and not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and hasattr(x, "dtype") and str(x.dtype).replace("torch.", "") != dtype:
        raise ValueError(f"{name} must be {dtype} (got {x.dtype})")
    if numel is not None and hasattr(x, "numel") and int(x.numel()) != int(numel):
        raise ValueError(f"{name} must have {numel} elements for these params (got {x.numel()})")
    if min_bytes is not None and hasattr(x, "numel") and hasattr(x, "element_size"):
        have = int(x.numel()) * int(x.element_size())
        if have < int(min_bytes):
            raise ValueError(f"{name} must hold at least {min_bytes} bytes (got {have})")
    return x.data_ptr()


def _sizes(params: Params):
    """Element counts of grad_out, weight and grad_in that ``params`` describe."""
    p = params
    return (p.batch * p.out_channels * p.out_h * p.out_w,
            p.out_channels * p.in_channels * p.kernel_h * p.kernel_w,
            p.batch * p.in_channels * p.in_h * p.in_w)


def _in_dtype(code: int) -> str | None:
    return _TORCH_DTYPE_NAME.get(int(code))


def _stream(stream) -> int | None:
    """The cudaStream_t of a torch stream (or an integer handle, passed through).
    A torch stream must belong to the current device."""
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    dev = getattr(stream, "device", None)
    index = getattr(dev, "index", None) if dev is not None else None
    if index is not None and int(index) != _current_device():
        raise ValueError(f"stream is on cuda:{index} but the current device is cuda:{_current_device()}")
    return stream.cuda_stream


def _check(rc: int, where: str) -> int:
    if rc != 0:
        raise DgradError(rc, where)
    return rc


def conv2d_grad_input(grad_out, weight, grad_in, params: Params, dtype: int, stream=None) -> None:
    n_go, n_w, n_gi = _sizes(params)
    rc = library().conv2d_grad_input(_addr(grad_out, "grad_out", _in_dtype(dtype), n_go),
                                     _addr(weight, "weight", _in_dtype(dtype), n_w),
                                     _addr(grad_in, "grad_in", "float32", n_gi),
                                     ctypes.byref(params), int(dtype), _stream(stream))
    _check(rc, "conv2d_grad_input")


def conv2d_grad_input_workspace_size(params: Params, dtype: int) -> int:
    return int(library().conv2d_grad_input_workspace_size(ctypes.byref(params), int(dtype)))


def conv2d_grad_input_pack_weight(weight, packed, packed_bytes: int, params: Params, dtype: int,
                                  stream=None) -> None:
    _, n_w, _ = _sizes(params)
    rc = library().conv2d_grad_input_pack_weight(_addr(weight, "weight", _in_dtype(dtype), n_w),
                                                 _addr(packed, "packed", min_bytes=int(packed_bytes)),
                                                 int(packed_bytes), ctypes.byref(params), int(dtype),
                                                 _stream(stream))
    _check(rc, "conv2d_grad_input_pack_weight")


def conv2d_grad_input_prepacked(grad_out, packed, grad_in, params: Params, dtype: int,
                                stream=None) -> None:
    """``packed``: the buffer conv2d_grad_input_pack_weight filled, or -- when
    the workspace size is 0 -- the weight tensor itself."""
    n_go, n_w, n_gi = _sizes(params)
    ws = conv2d_grad_input_workspace_size(params, dtype)
    packed_addr = (_addr(packed, "packed", min_bytes=ws) if ws > 0
                   else _addr(packed, "packed (the weight tensor)", _in_dtype(dtype), n_w))
    rc = library().conv2d_grad_input_prepacked(_addr(grad_out, "grad_out", _in_dtype(dtype), n_go),
                                               packed_addr,
                                               _addr(grad_in, "grad_in", "float32", n_gi),
                                               ctypes.byref(params), int(dtype), _stream(stream))
    _check(rc, "conv2d_grad_input_prepacked")


def conv2d_grad_input_check_errors(stream=None) -> int:
    """Returns the status (0, DGRAD_ERR_TIMEOUT = 6 or DGRAD_ERR_CUDA = 5) without raising."""
    return int(library().conv2d_grad_input_check_errors(_stream(stream)))


def conv2d_grad_input_status_string(status: int) -> str:
    return library().conv2d_grad_input_status_string(int(status)).decode()


def conv2d_grad_input_select_kernel(params: Params, dtype: int) -> int:
    """DGRAD_KERNEL_TC (1), DGRAD_KERNEL_SIMT (2) or DGRAD_KERNEL_TC_POSM (3), or a negative status."""
    return int(library().conv2d_grad_input_select_kernel(ctypes.byref(params), int(dtype)))


def conv2d_grad_input_set_kernel(kernel: int) -> int:
    return int(library().conv2d_grad_input_set_kernel(int(kernel)))


def conv2d_grad_input_set_wait_limit_ns(ns: int) -> int:
    return int(library().conv2d_grad_input_set_wait_limit_ns(int(ns)))


def conv2d_grad_input_set_debug(flags: int) -> int:
    return int(library().conv2d_grad_input_set_debug(int(flags)))


def conv2d_grad_input_noalloc(grad_out, weight, grad_in, params: Params, dtype: int,
                              stream=None) -> None:
    """conv2d_grad_input for callers that cannot allocate device memory.

    The packed weights go to a fixed 8 MiB array inside the library rather
    than a temporary allocation; calls that could overlap on the GPU must be
    ordered by the caller, and problems whose packed weights exceed 8 MiB
    raise DgradError(DGRAD_ERR_WORKSPACE).
    """
    n_go, n_w, n_gi = _sizes(params)
    rc = library().conv2d_grad_input_noalloc(_addr(grad_out, "grad_out", _in_dtype(dtype), n_go),
                                             _addr(weight, "weight", _in_dtype(dtype), n_w),
                                             _addr(grad_in, "grad_in", "float32", n_gi),
                                             ctypes.byref(params), int(dtype), _stream(stream))
    _check(rc, "conv2d_grad_input_noalloc")


def conv2d_forward(x, weight, out, params: Params, dtype: int, stream=None) -> None:
    """Forward convolution of the layer ``params`` describes (stride 1 to 8):
    x [N,Ci,H,W], weight [Co,Ci,kH,kW] -> out [N,Co,OH,OW] float32."""
    n_out, n_w, n_x = _sizes(params)
    rc = library().conv2d_forward(_addr(x, "x", _in_dtype(dtype), n_x),
                                  _addr(weight, "weight", _in_dtype(dtype), n_w),
                                  _addr(out, "out", "float32", n_out), ctypes.byref(params),
                                  int(dtype), _stream(stream))
    _check(rc, "conv2d_forward")


def _rms_args(x, w_norm, w_proj, c, params: RmsParams, dtype: int):
    m, n, k = int(params.m), int(params.n), int(params.k)
    t = _in_dtype(dtype)
    return (_addr(x, "x", t, m * k), _addr(w_norm, "w_norm", t, k), _addr(w_proj, "w_proj", t, k * n),
            _addr(c, "c", "float32", m * n))


def rmsnorm_matmul(x, w_norm, w_proj, c, params: RmsParams, dtype: int, stream=None) -> None:
    """C [m, n] = RmsNorm(X [m, k], W_norm [k]) x W_proj [k, n] (include/rmsnorm_matmul.h)."""
    rc = library().rmsnorm_matmul(*_rms_args(x, w_norm, w_proj, c, params, dtype), ctypes.byref(params),
                                  int(dtype), _stream(stream))
    _check(rc, "rmsnorm_matmul")


def rmsnorm_matmul_select_kernel(x, w_norm, w_proj, c, params: RmsParams, dtype: int) -> int:
    """DGRAD_KERNEL_TC (1) or DGRAD_KERNEL_SIMT (2) for these buffers, or a negative status."""
    return int(library().rmsnorm_matmul_select_kernel(*_rms_args(x, w_norm, w_proj, c, params, dtype),
                                                      ctypes.byref(params), int(dtype)))


def rmsnorm_matmul_set_kernel(kernel: int) -> int:
    return int(library().rmsnorm_matmul_set_kernel(int(kernel)))


def rmsnorm_matmul_check_errors(stream=None) -> int:
    """Returns the status (0, DGRAD_ERR_TIMEOUT = 6 or DGRAD_ERR_CUDA = 5) without raising."""
    return int(library().rmsnorm_matmul_check_errors(_stream(stream)))


def _mha_args(q, k, d_out, lse, dv, params: MhaParams, dtype: int):
    qs, nh, nkv, hd = int(params.q_seq), int(params.num_heads), int(params.num_kv_heads), int(params.head_dim)
    kv = qs if int(params.kv_seq) == 0 else int(params.kv_seq)
    t = _in_dtype(dtype)
    return (_addr(q, "q", t, qs * nh * hd), _addr(k, "k", t, kv * nkv * hd), _addr(d_out, "d_out", t, qs * nh * hd),
            _addr(lse, "lse", "float32", qs * nh * 2), _addr(dv, "dv", "float32", kv * nkv * hd))


def mha_grad_v(q, k, d_out, lse, dv, params: MhaParams, dtype: int, stream=None) -> None:
    """dV [kv, num_kv_heads, head_dim] of attention (include/mha_grad_v.h)."""
    rc = library().mha_grad_v(*_mha_args(q, k, d_out, lse, dv, params, dtype), ctypes.byref(params), int(dtype),
                              _stream(stream))
    _check(rc, "mha_grad_v")


def mha_grad_v_select_kernel(q, k, d_out, lse, dv, params: MhaParams, dtype: int) -> int:
    """DGRAD_KERNEL_TC (1) or DGRAD_KERNEL_SIMT (2) for these buffers, or a negative status."""
    return int(library().mha_grad_v_select_kernel(*_mha_args(q, k, d_out, lse, dv, params, dtype),
                                                  ctypes.byref(params), int(dtype)))


def mha_grad_v_set_kernel(kernel: int) -> int:
    return int(library().mha_grad_v_set_kernel(int(kernel)))


def mha_grad_v_check_errors(stream=None) -> int:
    """Returns the status (0, DGRAD_ERR_TIMEOUT = 6 or DGRAD_ERR_CUDA = 5) without raising."""
    return int(library().mha_grad_v_check_errors(_stream(stream)))
