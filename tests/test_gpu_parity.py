"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bar (element by element): max|gpu - oracle| / max|oracle| <= 2e-3 for bf16/fp16
inputs (the oracle is fed the identical rounded values) and <= 5e-3 for fp32
inputs on TF32 tensor cores; the CUDA-core kernel (float32 products) is held
to 1e-5.  The full-size workloads, element by element, are in
test_gpu_fullsize.py.
"""
import numpy as np
import pytest
import torch

import oracle
from conv2d_backward_implicit_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-3, "f16": 2e-3, "f32": 5e-3}
SIMT_TOL = 1e-5


@pytest.fixture(scope="module")
def dg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import conv2d_backward_implicit_gb300 as mod
    mod.library()
    return mod


@pytest.fixture(autouse=True)
def _reset_kernel_choice(request):
    yield
    if torch.cuda.is_available():
        import conv2d_backward_implicit_gb300 as mod
        mod.conv2d_grad_input_set_kernel(mod.DGRAD_KERNEL_AUTO)
        mod.conv2d_grad_input_set_debug(0)


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(got).all(), "non-finite output"
    denom = max(float(np.max(np.abs(ref))), 1e-30)
    return float(np.max(np.abs(got - ref))) / denom


def make_case(shape, dtype, seed):
    N, Ci, H, W, Co, kH, kW, s, ph, pw = shape
    OH, OW = oracle.out_size(H, kH, ph, s), oracle.out_size(W, kW, pw, s)
    wl = workloads.Workload(f"case{shape}", N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW, dtype,
                            "uniform")
    return wl


def run_gpu(dg, wl, g, w, kernel=None, via="call", stream=None):
    dev = torch.device("cuda")
    gd, wd = g.to(dev), w.to(dev)
    out = torch.full(wl.grad_in_shape, float("nan"), device=dev, dtype=torch.float32)
    p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    code = dg.DTYPE_CODE[wl.dtype]
    if kernel is not None:
        dg.conv2d_grad_input_set_kernel(kernel)
    st = stream or torch.cuda.current_stream()
    if via == "call":
        dg.conv2d_grad_input(gd, wd, out, p, code, st)
    else:
        ws = dg.conv2d_grad_input_workspace_size(p, code)
        if ws:
            packed = torch.empty(ws, dtype=torch.uint8, device=dev)
            dg.conv2d_grad_input_pack_weight(wd, packed, ws, p, code, st)
            dg.conv2d_grad_input_prepacked(gd, packed, out, p, code, st)
        else:
            dg.conv2d_grad_input_prepacked(gd, wd, out, p, code, st)
    rc = dg.conv2d_grad_input_check_errors(st)
    assert rc == 0, dg.conv2d_grad_input_status_string(rc)
    return out


def oracle_full(wl, g, w):
    return oracle.dgrad(g.double().numpy(), w.double().numpy(), wl.H, wl.W, wl.stride,
                        wl.padding_h, wl.padding_w)


# ------------------------------------------------------------ the workloads
REDUCED = {"tiny": 1, "resnet": 2, "strided": 2, "pointwise": 3, "stem": 1}


@pytest.mark.parametrize("key", list(REDUCED))
def test_workload_reduced_batch_tc(dg, key):
    wl = workloads.BY_KEY[key]
    wl = wl.with_batch(REDUCED[key]) if wl.N != REDUCED[key] else wl
    g, w = workloads.make_inputs(wl, seed=0)
    p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    assert dg.conv2d_grad_input_select_kernel(p, dg.DTYPE_CODE[wl.dtype]) == dg.DGRAD_KERNEL_TC
    out = run_gpu(dg, wl, g, w)
    err = rel_err(out.cpu().numpy(), oracle_full(wl, g, w))
    assert err <= TOL[wl.dtype], f"{wl.name}: {err:.3g}"


@pytest.mark.parametrize("key", list(REDUCED))
def test_workload_reduced_batch_simt(dg, key):
    wl = workloads.BY_KEY[key]
    wl = wl.with_batch(1)
    g, w = workloads.make_inputs(wl, seed=0)
    out = run_gpu(dg, wl, g, w, kernel=dg.DGRAD_KERNEL_SIMT)
    err = rel_err(out.cpu().numpy(), oracle_full(wl, g, w))
    assert err <= SIMT_TOL, f"{wl.name}: {err:.3g}"


# --------------------------------------------------------------- sweeps
TINY_SWEEP = workloads.random_small_shapes(60, seed=2024)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_small_shape_sweep_tc(dg, dtype):
    worst = 0.0
    for idx, shape in enumerate(TINY_SWEEP):
        wl = make_case(shape, dtype, idx)
        g, w = workloads.make_inputs(wl, seed=idx)
        out = run_gpu(dg, wl, g, w, kernel=dg.DGRAD_KERNEL_TC)
        err = rel_err(out.cpu().numpy(), oracle_full(wl, g, w))
        worst = max(worst, err)
        assert err <= TOL[dtype], f"{shape} {dtype}: {err:.3g}"
    print(f"worst {dtype}: {worst:.3g}")


def test_small_shape_sweep_simt(dg):
    for idx, shape in enumerate(TINY_SWEEP[:30]):
        wl = make_case(shape, "f32", idx)
        g, w = workloads.make_inputs(wl, seed=idx)
        out = run_gpu(dg, wl, g, w, kernel=dg.DGRAD_KERNEL_SIMT)
        err = rel_err(out.cpu().numpy(), oracle_full(wl, g, w))
        assert err <= SIMT_TOL, f"{shape}: {err:.3g}"


MEDIUM = workloads.random_small_shapes(24, seed=99, max_hw=37, max_c=80, max_k=7,
                                       strides=(1, 2, 3, 4))


@pytest.mark.parametrize("idx", range(len(MEDIUM)))
def test_medium_shape_sweep_tc(dg, idx):
    shape = MEDIUM[idx]
    dtype = ("bf16", "f16", "f32")[idx % 3]
    wl = make_case(shape, dtype, idx)
    g, w = workloads.make_inputs(wl, seed=500 + idx)
    out = run_gpu(dg, wl, g, w, kernel=dg.DGRAD_KERNEL_TC)
    err = rel_err(out.cpu().numpy(), oracle_full(wl, g, w))
    assert err <= TOL[dtype], f"{shape} {dtype}: {err:.3g}"


# ------------------------------------------------------------ edge cases
EDGE = {
    # (N, Ci, H, W, Co, kH, kW, s, ph, pw)
    "stride_above_kernel": (2, 5, 9, 10, 6, 1, 1, 3, 0, 0),
    "stride4_k2": (1, 7, 17, 13, 9, 2, 2, 4, 1, 0),
    "padding_at_kernel": (2, 3, 5, 6, 4, 3, 3, 1, 3, 2),
    "one_by_one_pad1": (1, 16, 7, 7, 32, 1, 1, 1, 1, 1),
    "off_centre_3x3_p0": (2, 16, 12, 12, 16, 3, 3, 1, 0, 0),
    "two_by_two_p0": (2, 8, 9, 9, 8, 2, 2, 1, 0, 0),
    "rect_kernel_pad_mismatch": (2, 12, 11, 15, 20, 5, 2, 2, 2, 0),
    "image_smaller_than_stride": (3, 4, 1, 2, 5, 3, 3, 3, 1, 1),
    "single_output": (2, 6, 3, 3, 5, 3, 3, 1, 0, 0),
    "ci_over_256": (1, 300, 6, 7, 40, 3, 3, 1, 1, 1),
    "co_not_multiple_of_chunk": (2, 24, 10, 9, 70, 3, 3, 2, 1, 1),
    "wide_rows": (1, 8, 4, 300, 16, 3, 3, 1, 1, 1),
    "ci_3_stem_like": (2, 3, 30, 30, 24, 7, 7, 2, 3, 3),
    "large_kernel_s1": (1, 16, 20, 20, 16, 7, 7, 1, 3, 3),
    "ragged_tail": (3, 40, 13, 17, 33, 3, 3, 1, 1, 1),
}


@pytest.mark.parametrize("name", sorted(EDGE))
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_edge_case_tc(dg, name, dtype):
    wl = make_case(EDGE[name], dtype, 0)
    g, w = workloads.make_inputs(wl, seed=sorted(EDGE).index(name))
    p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    assert dg.conv2d_grad_input_select_kernel(p, dg.DTYPE_CODE[dtype]) == dg.DGRAD_KERNEL_TC
    out = run_gpu(dg, wl, g, w)
    err = rel_err(out.cpu().numpy(), oracle_full(wl, g, w))
    assert err <= TOL[dtype], f"{name}: {err:.3g}"


def test_zero_filled_phases_are_exact_zero(dg):
    # Stride 3 with a 1x1 kernel: 8 of the 9 phases receive no tap.
    wl = make_case((2, 4, 9, 9, 5, 1, 1, 3, 0, 0), "bf16", 0)
    g, w = workloads.make_inputs(wl, seed=3)
    out = run_gpu(dg, wl, g, w).cpu().numpy()
    mask = np.ones((9, 9), dtype=bool)
    mask[::3, ::3] = False
    assert np.all(out[:, :, mask] == 0.0)


# ----------------------------------------------------- buffers and streams
def test_guard_bands_untouched(dg):
    wl = make_case((2, 20, 11, 9, 24, 3, 3, 2, 1, 1), "bf16", 0)
    g, w = workloads.make_inputs(wl, seed=5)
    dev = torch.device("cuda")
    n = int(np.prod(wl.grad_in_shape))
    guard = 4096
    buf = torch.full((n + 2 * guard,), 1234.5, device=dev, dtype=torch.float32)
    out = buf[guard:guard + n].view(wl.grad_in_shape)
    p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    for kernel in (dg.DGRAD_KERNEL_TC, dg.DGRAD_KERNEL_SIMT):
        dg.conv2d_grad_input_set_kernel(kernel)
        dg.conv2d_grad_input(g.to(dev), w.to(dev), out, p, dg.DGRAD_BF16)
        assert dg.conv2d_grad_input_check_errors() == 0
        b = buf.cpu()
        assert torch.all(b[:guard] == 1234.5) and torch.all(b[guard + n:] == 1234.5)
        err = rel_err(out.cpu().numpy(), oracle_full(wl, g, w))
        assert err <= TOL["bf16"]


def test_grad_in_only_4_byte_aligned(dg):
    # grad_in needs only element (4-byte) alignment; the kernel must not use
    # wider stores when the buffer is not 8-byte aligned.
    wl = workloads.RESNET.with_batch(1)
    g, w = workloads.make_inputs(wl, seed=4)
    dev = torch.device("cuda")
    n = int(np.prod(wl.grad_in_shape))
    buf = torch.full((n + 1,), 5.0, device=dev, dtype=torch.float32)
    out = buf[1:].view(wl.grad_in_shape)
    assert out.data_ptr() % 8 == 4
    p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    dg.conv2d_grad_input(g.to(dev), w.to(dev), out, p, dg.DGRAD_BF16)
    assert dg.conv2d_grad_input_check_errors() == 0
    assert buf[0].item() == 5.0
    assert rel_err(out.cpu().numpy(), oracle_full(wl, g, w)) <= TOL["bf16"]


def test_deterministic_and_nondefault_stream(dg):
    wl = workloads.RESNET.with_batch(3)
    g, w = workloads.make_inputs(wl, seed=1)
    s = torch.cuda.Stream()
    a = run_gpu(dg, wl, g, w, stream=s)
    b = run_gpu(dg, wl, g, w)
    assert torch.equal(a, b)


def test_pack_reuse_across_inputs(dg):
    wl = workloads.STRIDED.with_batch(1)
    g1, w = workloads.make_inputs(wl, seed=1)
    g2, _ = workloads.make_inputs(wl, seed=2)
    dev = torch.device("cuda")
    p = dg.params_from_shapes(g1.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    ws = dg.conv2d_grad_input_workspace_size(p, dg.DGRAD_BF16)
    assert ws > 0
    packed = torch.empty(ws, dtype=torch.uint8, device=dev)
    dg.conv2d_grad_input_pack_weight(w.to(dev), packed, ws, p, dg.DGRAD_BF16)
    for g in (g1, g2):
        out = torch.empty(wl.grad_in_shape, device=dev)
        dg.conv2d_grad_input_prepacked(g.to(dev), packed, out, p, dg.DGRAD_BF16)
        assert dg.conv2d_grad_input_check_errors() == 0
        assert rel_err(out.cpu().numpy(), oracle_full(wl, g, w)) <= TOL["bf16"]


def test_argument_errors_leave_output_untouched(dg):
    wl = workloads.TINY
    g, w = workloads.make_inputs(wl, seed=0)
    dev = torch.device("cuda")
    gd, wd = g.to(dev), w.to(dev)
    out = torch.full(wl.grad_in_shape, 7.0, device=dev)
    bad = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h,
                                wl.padding_w)
    bad.out_h = 9  # off the formula
    # The binding refuses tensors whose sizes disagree with the params ...
    with pytest.raises(ValueError, match="elements"):
        dg.conv2d_grad_input(gd, wd, out, bad, dg.DGRAD_F32)
    # ... and the library itself checks the params (raw addresses pass the binding unchecked).
    with pytest.raises(dg.DgradError) as ei:
        dg.conv2d_grad_input(gd.data_ptr(), wd.data_ptr(), out.data_ptr(), bad, dg.DGRAD_F32)
    assert ei.value.status == 2
    good = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h,
                                 wl.padding_w)
    raw = torch.empty(g.numel() + 1, device=dev)
    with pytest.raises(dg.DgradError) as ei:
        dg.conv2d_grad_input(raw.data_ptr() + 2, wd, out, good, dg.DGRAD_F32)
    assert ei.value.status == 3
    small = torch.empty(16, dtype=torch.uint8, device=dev)
    with pytest.raises(dg.DgradError) as ei:
        dg.conv2d_grad_input_pack_weight(wd, small, 16, good, dg.DGRAD_F32)
    assert ei.value.status == 7
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
    assert dg.conv2d_grad_input_check_errors() == 0
