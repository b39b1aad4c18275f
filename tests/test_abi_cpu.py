"""The C-ABI library on the host: it loads, exports every declared symbol, and
rejects bad arguments before any device work (no GPU needed)."""
import ctypes
import os
import re

import pytest

import conv2d_backward_implicit_gb300 as dg
from conv2d_backward_implicit_gb300 import build_ext, workloads

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADER = os.path.join(INCLUDE, "conv2d_grad_input.h")


@pytest.fixture(scope="module")
def lib():
    if build_ext.is_stale():
        build_ext.build()
    return dg.library()


def declared_functions():
    """Every function declared in include/*.h (a return type, a name, an open parenthesis)."""
    names = set()
    for h in sorted(os.listdir(INCLUDE)):
        if not h.endswith(".h"):
            continue
        text = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, h)).read(), flags=re.S)
        names.update(re.findall(r"^\s*(?:const\s+)?(?:int|size_t|void|uint64_t|const char)\s*\*?\s*"
                                r"([a-z_0-9]+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_abi():
    names = declared_functions()
    for must in ("conv2d_grad_input", "conv2d_grad_input_workspace_size",
                 "conv2d_grad_input_pack_weight", "conv2d_grad_input_prepacked",
                 "conv2d_grad_input_check_errors", "conv2d_grad_input_status_string",
                 "conv2d_grad_input_noalloc", "conv2d_forward", "rmsnorm_matmul",
                 "rmsnorm_matmul_select_kernel", "rmsnorm_matmul_set_kernel",
                 "rmsnorm_matmul_check_errors"):
        assert must in names, must


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def params(wl):
    return dg.Params(wl.N, wl.Ci, wl.H, wl.W, wl.Co, wl.kH, wl.kW, wl.stride, wl.padding_h,
                     wl.OH, wl.OW, wl.padding_w)


def test_workloads_select_tensor_cores(lib):
    for wl in workloads.ALL:
        assert dg.conv2d_grad_input_select_kernel(params(wl), dg.DTYPE_CODE[wl.dtype]) == \
            dg.DGRAD_KERNEL_TC, wl.name


def test_workspace_sizes_closed_form(lib):
    # Packed weights hold each (tap, co, ci) product once, Ci padded to a whole 64-row
    # (Ci <= 64) or 128-row tile and Co to whole 128-byte rows (64 bf16/fp16 or 32 fp32):
    # none for the ResNet layer (16-bit, stride 1, weights resident in shared memory:
    # the kernel packs them there itself);
    # 9 taps (over 4 phases) x 256 x 128 bf16; 1024 x 256 fp16;
    # stem (stacked phases): 4 x 4 window taps (the union of the phases' tap
    # offsets) x 64 co x 16 columns (4 phases x 3 ci, padded to 16) fp32;
    # 9 x 32 (16 padded) x 64 (8 padded) fp32.
    want = {"resnet": 0, "strided": 9 * 256 * 128 * 2, "pointwise": 1024 * 256 * 2,
            "stem": 16 * 64 * 16 * 4, "tiny": 9 * 32 * 64 * 4}
    for key, nbytes in want.items():
        wl = workloads.BY_KEY[key]
        assert dg.conv2d_grad_input_workspace_size(params(wl), dg.DTYPE_CODE[wl.dtype]) == nbytes


def test_shape_validation(lib):
    wl = workloads.RESNET
    p = params(wl)
    code = dg.DGRAD_BF16
    for field, value, status in [("out_h", 55, 2), ("out_w", 57, 2), ("batch", 0, 2),
                                 ("stride", 0, 2), ("kernel_h", 0, 2), ("in_channels", 0, 2),
                                 ("kernel_w", 60, 2), ("padding_h", 2, 2)]:
        q = dg.Params(*[getattr(p, f) for f in dg.PARAM_FIELDS])
        setattr(q, field, value)
        assert dg.conv2d_grad_input_select_kernel(q, code) == -status, field
        assert dg.conv2d_grad_input_workspace_size(q, code) == 0
    assert dg.conv2d_grad_input_select_kernel(p, 9) == -1
    huge = dg.Params(*[getattr(p, f) for f in dg.PARAM_FIELDS])
    huge.batch = 1 << 30
    assert dg.conv2d_grad_input_select_kernel(huge, code) == -4


def test_null_and_bad_arguments_fail_on_the_host(lib):
    p = params(workloads.TINY)
    assert lib.conv2d_grad_input(None, None, None, ctypes.byref(p), 0, None) == 1
    bad = params(workloads.TINY)
    bad.out_w = 3
    # Valid-looking (never dereferenced) addresses: validation rejects before any CUDA call.
    assert lib.conv2d_grad_input(16, 16, 16, ctypes.byref(bad), 0, None) == 2
    assert lib.conv2d_grad_input(16, 16, 16, ctypes.byref(p), 7, None) == 1
    assert lib.conv2d_grad_input(18, 16, 16, ctypes.byref(p), 0, None) == 3
    assert lib.conv2d_grad_input_prepacked(16, None, 16, ctypes.byref(p), 0, None) == 1
    assert lib.conv2d_grad_input_pack_weight(16, 16, 8, ctypes.byref(p), 0, None) == 7


def test_status_strings_and_settings(lib):
    assert dg.conv2d_grad_input_status_string(0) == "ok"
    assert dg.conv2d_grad_input_status_string(6) == "device wait timed out"
    assert dg.conv2d_grad_input_status_string(99) == "unknown status"
    prev = dg.conv2d_grad_input_set_kernel(dg.DGRAD_KERNEL_SIMT)
    assert prev == dg.DGRAD_KERNEL_AUTO
    assert dg.conv2d_grad_input_select_kernel(params(workloads.RESNET), 1) == dg.DGRAD_KERNEL_SIMT
    assert dg.conv2d_grad_input_workspace_size(params(workloads.RESNET), 1) == 0
    assert dg.conv2d_grad_input_set_kernel(dg.DGRAD_KERNEL_AUTO) == dg.DGRAD_KERNEL_SIMT
    assert dg.conv2d_grad_input_set_kernel(5) < 0
    old = dg.conv2d_grad_input_set_wait_limit_ns(1000)
    assert dg.conv2d_grad_input_set_wait_limit_ns(0) == 1000
    assert old == 2_000_000_000
    assert dg.conv2d_grad_input_set_debug(0) == 0


def test_positions_on_m_selection(lib):
    prev = dg.conv2d_grad_input_set_kernel(dg.DGRAD_KERNEL_TC_POSM)
    try:
        assert dg.conv2d_grad_input_select_kernel(params(workloads.RESNET), 1) == dg.DGRAD_KERNEL_TC_POSM
        assert dg.conv2d_grad_input_select_kernel(params(workloads.RESNET), 2) == dg.DGRAD_KERNEL_TC_POSM
        # fp32, Ci > 64 and stride 2 stay with the general tensor-core mode
        assert dg.conv2d_grad_input_select_kernel(params(workloads.RESNET), 0) == dg.DGRAD_KERNEL_TC
        assert dg.conv2d_grad_input_select_kernel(params(workloads.STRIDED), 1) == dg.DGRAD_KERNEL_TC
        assert dg.conv2d_grad_input_select_kernel(params(workloads.POINTWISE), 2) == dg.DGRAD_KERNEL_TC
        # same packed weights as the general mode
        assert dg.conv2d_grad_input_workspace_size(params(workloads.RESNET), 1) == 9 * 64 * 64 * 2
    finally:
        dg.conv2d_grad_input_set_kernel(prev)
    assert dg.conv2d_grad_input_select_kernel(params(workloads.RESNET), 1) == dg.DGRAD_KERNEL_TC


def test_stride_above_four_uses_cuda_cores(lib):
    p = dg.Params(1, 4, 20, 20, 4, 3, 3, 5, 1, 4, 4, 1)
    assert dg.conv2d_grad_input_select_kernel(p, 0) == dg.DGRAD_KERNEL_SIMT


def test_forward_rejects_what_it_does_not_run(lib):
    # Stride above 8, or padding above kernel - 1 at stride 1: unsupported,
    # before any device work (the pointers are never touched).
    p = dg.Params(2, 16, 40, 40, 24, 3, 3, 9, 1, 5, 5, 1)
    assert lib.conv2d_forward(16, 16, 16, ctypes.byref(p), dg.DGRAD_BF16, None) == 4
    p = dg.Params(2, 16, 10, 10, 24, 3, 3, 1, 3, 14, 14, 3)
    assert lib.conv2d_forward(16, 16, 16, ctypes.byref(p), dg.DGRAD_BF16, None) == 4
    # An inconsistent layer is a shape error, as for the input gradient.
    p = dg.Params(2, 16, 10, 10, 24, 3, 3, 1, 1, 9, 10, 1)
    assert lib.conv2d_forward(16, 16, 16, ctypes.byref(p), dg.DGRAD_BF16, None) == 2
    assert lib.conv2d_forward(None, 16, 16, ctypes.byref(p), dg.DGRAD_BF16, None) == 1


def test_in_kernel_weight_pack_selection(lib):
    # The kernel packs the weights itself (workspace 0) exactly for 16-bit
    # stride-1 tensor-core plans whose packed weights stay resident in shared
    # memory; fp32 (TF32 rounding), strided layers and streamed weights keep
    # the pack kernel and its workspace.
    def params_of(shape):
        N, Ci, H, W, Co, kH, kW, s, ph, pw = shape
        oh, ow = (H + 2 * ph - kH) // s + 1, (W + 2 * pw - kW) // s + 1
        return dg.Params(N, Ci, H, W, Co, kH, kW, s, ph, oh, ow, pw)

    def ws(shape, code):
        return dg.conv2d_grad_input_workspace_size(params_of(shape), code)
    packed_in_kernel = [(32, 64, 56, 56, 64, 3, 3, 1, 1, 1),   # the ResNet layer (64-wide frame)
                        (3, 40, 13, 17, 33, 3, 3, 1, 1, 1),     # odd width: the general frame
                        (2, 6, 3, 3, 5, 3, 3, 1, 0, 0)]
    for shape in packed_in_kernel:
        for code in (dg.DGRAD_BF16, dg.DGRAD_F16):
            assert dg.conv2d_grad_input_select_kernel(params_of(shape), code) == dg.DGRAD_KERNEL_TC
            assert ws(shape, code) == 0, shape
        assert ws(shape, dg.DGRAD_F32) > 0, shape
    assert ws((32, 128, 56, 56, 256, 3, 3, 2, 1, 1), dg.DGRAD_BF16) > 0      # stride 2
    for streamed in [(1, 1024, 8, 8, 1024, 3, 3, 1, 1, 1), (1, 8, 4, 300, 16, 3, 3, 1, 1, 1),
                     (1, 64, 28, 112, 64, 3, 3, 1, 1, 1), (1, 16, 20, 20, 16, 7, 7, 1, 3, 3)]:
        assert ws(streamed, dg.DGRAD_BF16) > 0, streamed                     # streamed weights


def test_kernel_fingerprint_ignores_comments():
    import bench
    code = "int a; // note\n/* block\n comment */\nint b;  \n\n"
    assert bench.code_of(code) == "int a;\nint b;"
    assert bench.code_of(code) == bench.code_of(code.replace("note", "other note"))
    assert bench.code_of(code) != bench.code_of(code.replace("int b", "int c"))


def test_planner_accepts_every_valid_shape(lib):
    # Host-side planning over a random sweep of valid layers (strides 1-6,
    # kernels 1-7, paddings up to past the kernel, channels 1-300, all three
    # dtypes): every call plans a kernel -- tensor-core, or the CUDA-core
    # fallback -- never an error, and only tensor-core plans can ask for a
    # workspace.
    import random
    rng = random.Random(20240611)
    for _ in range(1500):
        s = rng.choice([1, 1, 2, 2, 3, 4, 5, 6])
        kH, kW = rng.randint(1, 7), rng.randint(1, 7)
        ph, pw = rng.randint(0, kH), rng.randint(0, kW)
        H = rng.randint(max(1, kH - 2 * ph), 80)
        W = rng.randint(max(1, kW - 2 * pw), 80)
        N, Ci, Co = rng.randint(1, 4), rng.randint(1, 300), rng.randint(1, 300)
        oh, ow = (H + 2 * ph - kH) // s + 1, (W + 2 * pw - kW) // s + 1
        p = dg.Params(N, Ci, H, W, Co, kH, kW, s, ph, oh, ow, pw)
        for code in (dg.DGRAD_F32, dg.DGRAD_BF16, dg.DGRAD_F16):
            k = dg.conv2d_grad_input_select_kernel(p, code)
            assert k in (dg.DGRAD_KERNEL_TC, dg.DGRAD_KERNEL_SIMT), (p, code, k)
            if k == dg.DGRAD_KERNEL_SIMT:
                assert dg.conv2d_grad_input_workspace_size(p, code) == 0


class _FakeCudaTensor:
    """Just enough of a tensor for the binding's host-side checks."""

    def __init__(self, dtype="bfloat16", contiguous=True, device="cuda", numel=None, index=None):
        self.dtype = f"torch.{dtype}"
        self.device = type("Dev", (), {"type": device, "index": index,
                                       "__str__": lambda s: device})()
        self._contiguous = contiguous
        self._numel = numel
        if numel is None:  # no size known: the size checks are skipped
            del self.__dict__["_numel"]

    def is_contiguous(self):
        return self._contiguous

    def data_ptr(self):
        return 1 << 20

    def __getattr__(self, name):
        if name in ("numel", "element_size") and "_numel" in self.__dict__:
            esize = 4 if "32" in self.dtype else (1 if "uint8" in self.dtype else 2)
            return (lambda: self._numel) if name == "numel" else (lambda: esize)
        raise AttributeError(name)


def test_binding_checks_tensors_before_calling_the_library(lib, monkeypatch):
    import torch
    import conv2d_backward_implicit_gb300.binding as binding
    monkeypatch.setattr(binding, "_current_device", lambda: 0)
    wl = workloads.RESNET
    p = params(wl)
    n_go = wl.N * wl.Co * wl.OH * wl.OW
    n_w = wl.Co * wl.Ci * wl.kH * wl.kW
    n_gi = wl.N * wl.Ci * wl.H * wl.W
    good_g, good_w = _FakeCudaTensor(), _FakeCudaTensor()
    out = _FakeCudaTensor("float32")
    cases = [
        (torch.zeros(4), good_w, out, "CUDA tensor"),                       # host memory
        (_FakeCudaTensor(contiguous=False), good_w, out, "contiguous"),     # a strided view
        (good_g, _FakeCudaTensor("float16"), out, "bfloat16"),              # dtype vs code
        (good_g, good_w, _FakeCudaTensor("bfloat16"), "float32"),           # grad_in is fp32
        # tensors smaller (or larger) than the params describe never reach a kernel
        (_FakeCudaTensor(numel=n_go - 1), good_w, out, "elements"),
        (good_g, _FakeCudaTensor(numel=n_w // 2), out, "elements"),
        (good_g, good_w, _FakeCudaTensor("float32", numel=n_gi - 56), "elements"),
        (good_g, good_w, _FakeCudaTensor("float32", numel=n_gi + 1), "elements"),
        # a tensor on another GPU than the current one
        (_FakeCudaTensor(index=1), good_w, out, "current device"),
        (good_g, good_w, _FakeCudaTensor("float32", index=3), "current device"),
    ]
    for g, w, o, msg in cases:
        with pytest.raises(ValueError, match=msg):
            dg.conv2d_grad_input(g, w, o, p, dg.DGRAD_BF16)
        with pytest.raises(ValueError, match=msg):
            dg.conv2d_grad_input_noalloc(g, w, o, p, dg.DGRAD_BF16)
        with pytest.raises(ValueError, match=msg):
            dg.conv2d_grad_input_prepacked(g, w, o, p, dg.DGRAD_BF16)  # ResNet packs in the kernel
    with pytest.raises(ValueError, match="CUDA tensor"):
        dg.conv2d_grad_input_prepacked(good_g, torch.zeros(4), out, p, dg.DGRAD_BF16)
    with pytest.raises(ValueError, match="float32"):
        dg.conv2d_forward(good_g, good_w, _FakeCudaTensor("float16"), p, dg.DGRAD_BF16)
    with pytest.raises(ValueError, match="elements"):
        dg.conv2d_forward(_FakeCudaTensor(numel=n_gi - 1), good_w, out, p, dg.DGRAD_BF16)
    # A packed-weight buffer smaller than the workspace the layer needs.
    s = params(workloads.STRIDED)
    ws = dg.conv2d_grad_input_workspace_size(s, dg.DGRAD_BF16)
    assert ws > 0
    with pytest.raises(ValueError, match="bytes"):
        dg.conv2d_grad_input_prepacked(good_g, _FakeCudaTensor("uint8", numel=ws - 16), out, s,
                                       dg.DGRAD_BF16)
    with pytest.raises(ValueError, match="bytes"):
        dg.conv2d_grad_input_pack_weight(good_w, _FakeCudaTensor("uint8", numel=ws - 1), ws, s,
                                         dg.DGRAD_BF16)
    # A stream of another device.
    other = type("S", (), {"device": type("D", (), {"index": 2})(), "cuda_stream": 0})()
    with pytest.raises(ValueError, match="stream"):
        dg.conv2d_grad_input(good_g, good_w, out, p, dg.DGRAD_BF16, other)


# ---------------------------------------------------------------- rmsnorm_matmul (host logic)
def test_rmsnorm_matmul_selection_and_validation(lib):
    sel = dg.rmsnorm_matmul_select_kernel
    A, W, B, C = 0x10000, 0x20000, 0x30000, 0x40000  # 16-byte aligned raw addresses
    p = dg.RmsParams(300, 320, 520, 1e-5)
    assert sel(A, W, B, C, p, dg.DGRAD_BF16) == dg.DGRAD_KERNEL_TC
    assert sel(A, W, B, C, p, dg.DGRAD_F16) == dg.DGRAD_KERNEL_TC
    assert sel(A, W, B, C, p, dg.DGRAD_F32) == dg.DGRAD_KERNEL_SIMT      # float32: CUDA cores
    assert sel(A, W, B, C + 4, p, dg.DGRAD_BF16) == dg.DGRAD_KERNEL_SIMT  # C off 16 bytes
    assert sel(A + 2, W, B, C, p, dg.DGRAD_BF16) == dg.DGRAD_KERNEL_SIMT  # X off 16 bytes
    assert sel(A, W, B, C, dg.RmsParams(300, 330, 520, 1e-5), dg.DGRAD_BF16) == dg.DGRAD_KERNEL_SIMT
    assert sel(A, W, B, C, dg.RmsParams(300, 320, 521, 1e-5), dg.DGRAD_BF16) == dg.DGRAD_KERNEL_SIMT
    assert sel(0, W, B, C, p, dg.DGRAD_BF16) == -1                        # NULL
    assert sel(A, W, B, C, p, 7) == -1                                    # dtype
    assert sel(A, W, B, C, dg.RmsParams(300, 320, 520, -1.0), dg.DGRAD_BF16) == -1
    assert sel(A, W, B, C, dg.RmsParams(300, 320, 520, float("nan")), dg.DGRAD_BF16) == -1
    assert sel(A, W, B, C, dg.RmsParams(0, 320, 520, 0.0), dg.DGRAD_BF16) == -2
    assert sel(A + 1, W, B, C, p, dg.DGRAD_BF16) == -3                    # element alignment
    assert sel(A, W, B, C + 2, p, dg.DGRAD_F32) == -3
    assert sel(A, W, B, C, dg.RmsParams(1 << 16, 1 << 16, 8, 0.0), dg.DGRAD_BF16) == -4  # 2^32 outputs
    assert dg.rmsnorm_matmul_set_kernel(dg.DGRAD_KERNEL_TC) == dg.DGRAD_KERNEL_AUTO
    try:
        assert sel(A, W, B, C, p, dg.DGRAD_BF16) == dg.DGRAD_KERNEL_TC
        assert sel(A, W, B, C, p, dg.DGRAD_F32) == -4                     # forced but not applicable
        assert dg.rmsnorm_matmul_set_kernel(dg.DGRAD_KERNEL_SIMT) == dg.DGRAD_KERNEL_TC
        assert sel(A, W, B, C, p, dg.DGRAD_BF16) == dg.DGRAD_KERNEL_SIMT
        assert dg.rmsnorm_matmul_set_kernel(3) == 1                       # DGRAD_ERR_INVALID_ARG
    finally:
        dg.rmsnorm_matmul_set_kernel(dg.DGRAD_KERNEL_AUTO)


def test_rmsnorm_matmul_binding_checks_tensors(lib, monkeypatch):
    """Sizes, dtypes and devices of the four buffers are checked on the host
    before the library is called (fake CUDA tensors: nothing reaches a GPU)."""
    import torch
    import conv2d_backward_implicit_gb300.binding as binding
    monkeypatch.setattr(binding, "_current_device", lambda: 0)
    p = dg.RmsParams(4, 64, 8, 0.0)
    x = _FakeCudaTensor(numel=32)
    wn = _FakeCudaTensor(numel=8)
    wp = _FakeCudaTensor(numel=512)
    c = _FakeCudaTensor("float32", numel=256)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dg.rmsnorm_matmul(torch.zeros(4, 8, dtype=torch.bfloat16), wn, wp, c, p, dg.DGRAD_BF16)
    for bad, what in (((_FakeCudaTensor(numel=33), wn, wp, c), "x must have 32"),
                      ((x, _FakeCudaTensor(numel=9), wp, c), "w_norm must have 8"),
                      ((x, wn, _FakeCudaTensor(numel=511), c), "w_proj must have 512"),
                      ((x, wn, wp, _FakeCudaTensor("float32", numel=255)), "c must have 256"),
                      ((x, wn, wp, _FakeCudaTensor("bfloat16", numel=256)), "float32"),
                      ((_FakeCudaTensor("float16", numel=32), wn, wp, c), "bfloat16"),
                      ((x, wn, wp, _FakeCudaTensor("float32", numel=256, index=1)), "current device")):
        with pytest.raises(ValueError, match=what):
            dg.rmsnorm_matmul(*bad, p, dg.DGRAD_BF16)


# ---------------------------------------------------------------- mha_grad_v (host logic)
def test_mha_grad_v_validation_and_selection(lib):
    sel = dg.mha_grad_v_select_kernel
    Q, K, O, L, V = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000
    p = dg.MhaParams(128, 0, 8, 2, 64, 0)
    assert sel(Q, K, O, L, V, p, dg.DGRAD_F32) == dg.DGRAD_KERNEL_SIMT
    assert sel(0, K, O, L, V, p, dg.DGRAD_BF16) == -1                          # NULL
    assert sel(Q, K, O, L, V, p, 9) == -1                                      # dtype
    assert sel(Q, K, O, L, V, dg.MhaParams(0, 0, 8, 2, 64, 0), dg.DGRAD_BF16) == -2
    assert sel(Q, K, O, L, V, dg.MhaParams(128, 0, 6, 4, 64, 0), dg.DGRAD_BF16) == -2   # 6 % 4
    assert sel(Q, K, O, L, V, dg.MhaParams(128, 0, 8, 2, 0, 0), dg.DGRAD_BF16) == -2
    assert sel(Q + 1, K, O, L, V, p, dg.DGRAD_BF16) == -3                      # element alignment
    assert sel(Q, K, O, L + 2, V, p, dg.DGRAD_BF16) == -3
    assert sel(Q, K, O, L, V, dg.MhaParams(128, 0, 8, 2, 512, 0), dg.DGRAD_BF16) == -4  # head_dim
    assert sel(Q, K, O, L, V, p, dg.DGRAD_BF16) == dg.DGRAD_KERNEL_TC
    assert sel(Q, K, O, L, V, p, dg.DGRAD_F16) == dg.DGRAD_KERNEL_TC
    assert sel(Q, K, O, L, V, dg.MhaParams(128, 0, 3, 1, 64, 0), dg.DGRAD_BF16) == dg.DGRAD_KERNEL_SIMT  # odd heads
    assert sel(Q, K, O, L + 8, V, p, dg.DGRAD_BF16) == dg.DGRAD_KERNEL_SIMT    # LSE not 16-byte aligned
    assert sel(Q, K, O, L, V, dg.MhaParams(128, 0, 8, 2, 32, 0), dg.DGRAD_BF16) == dg.DGRAD_KERNEL_SIMT  # head_dim
    assert dg.mha_grad_v_set_kernel(dg.DGRAD_KERNEL_SIMT) == dg.DGRAD_KERNEL_AUTO
    try:
        assert sel(Q, K, O, L, V, p, dg.DGRAD_BF16) == dg.DGRAD_KERNEL_SIMT
        assert dg.mha_grad_v_set_kernel(dg.DGRAD_KERNEL_TC) == dg.DGRAD_KERNEL_SIMT
        assert sel(Q, K, O, L, V, p, dg.DGRAD_F32) == -4                       # forced, not applicable
        assert dg.mha_grad_v_set_kernel(7) == 1
    finally:
        dg.mha_grad_v_set_kernel(dg.DGRAD_KERNEL_AUTO)


def test_mha_grad_v_binding_checks_tensors(lib, monkeypatch):
    import conv2d_backward_implicit_gb300.binding as binding
    monkeypatch.setattr(binding, "_current_device", lambda: 0)
    p = dg.MhaParams(10, 0, 4, 2, 8, 0)   # kv = 10
    q = _FakeCudaTensor(numel=320)
    k = _FakeCudaTensor(numel=160)
    go = _FakeCudaTensor(numel=320)
    lse = _FakeCudaTensor("float32", numel=80)
    dv = _FakeCudaTensor("float32", numel=160)
    for bad, what in (((_FakeCudaTensor(numel=321), k, go, lse, dv), "q must have 320"),
                      ((q, _FakeCudaTensor(numel=159), go, lse, dv), "k must have 160"),
                      ((q, k, _FakeCudaTensor(numel=10), lse, dv), "d_out must have 320"),
                      ((q, k, go, _FakeCudaTensor("float32", numel=40), dv), "lse must have 80"),
                      ((q, k, go, lse, _FakeCudaTensor("bfloat16", numel=160)), "float32"),
                      ((q, k, go, lse, _FakeCudaTensor("float32", numel=160, index=3)), "current device")):
        with pytest.raises(ValueError, match=what):
            dg.mha_grad_v(*bad, p, dg.DGRAD_BF16)
