"""GPU parity of the positions-on-M tensor-core mode (DGRAD_KERNEL_TC_POSM)
against the CPU oracle: the ResNet workload (reduced batch element by
element, full size on sampled points), shapes at the edges of the mode's
range, the fallback to the general mode for a grad_out pointer the TMA gather
cannot use, and the timeout path.  Same bar as the general mode:
max|gpu - oracle| / max|oracle| <= 2e-3 for bf16 / fp16 inputs."""
import numpy as np
import pytest
import torch

import oracle
from conv2d_backward_implicit_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def dg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import conv2d_backward_implicit_gb300 as mod
    mod.library()
    return mod


@pytest.fixture(autouse=True)
def _posm(request):
    if torch.cuda.is_available():
        import conv2d_backward_implicit_gb300 as mod
        mod.conv2d_grad_input_set_kernel(mod.DGRAD_KERNEL_TC_POSM)
    yield
    if torch.cuda.is_available():
        import conv2d_backward_implicit_gb300 as mod
        mod.conv2d_grad_input_set_kernel(mod.DGRAD_KERNEL_AUTO)
        mod.conv2d_grad_input_set_debug(0)
        mod.conv2d_grad_input_set_wait_limit_ns(0)


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(got).all(), "non-finite output"
    return float(np.max(np.abs(got - ref))) / max(float(np.max(np.abs(ref))), 1e-30)


def case(shape, dtype):
    N, Ci, H, W, Co, kH, kW, s, ph, pw = shape
    OH, OW = oracle.out_size(H, kH, ph, s), oracle.out_size(W, kW, pw, s)
    return workloads.Workload(f"case{shape}", N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW, dtype,
                              "uniform")


def params(dg, wl, g, w):
    return dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h,
                                 wl.padding_w)


def run(dg, wl, g, w, via="call", g_offset=0):
    dev = torch.device("cuda")
    if g_offset:
        # grad_out at an element offset inside a larger buffer
        flat = torch.zeros(g.numel() + g_offset, dtype=g.dtype, device=dev)
        flat[g_offset:] = g.reshape(-1).to(dev)
        gd = flat[g_offset:].view(g.shape)
    else:
        gd = g.to(dev)
    wd = w.to(dev)
    out = torch.full(wl.grad_in_shape, float("nan"), device=dev)
    p = params(dg, wl, g, w)
    code = dg.DTYPE_CODE[wl.dtype]
    if via == "call":
        dg.conv2d_grad_input(gd, wd, out, p, code)
    else:
        ws = dg.conv2d_grad_input_workspace_size(p, code)
        if ws:
            packed = torch.empty(ws, dtype=torch.uint8, device=dev)
            dg.conv2d_grad_input_pack_weight(wd, packed, ws, p, code)
            dg.conv2d_grad_input_prepacked(gd, packed, out, p, code)
        else:  # the kernel packs the weights itself
            dg.conv2d_grad_input_prepacked(gd, wd, out, p, code)
    rc = dg.conv2d_grad_input_check_errors()
    assert rc == 0, dg.conv2d_grad_input_status_string(rc)
    return out


def full_oracle(wl, g, w):
    return oracle.dgrad(g.double().numpy(), w.double().numpy(), wl.H, wl.W, wl.stride,
                        wl.padding_h, wl.padding_w)


def test_resnet_reduced_batch(dg):
    wl = workloads.RESNET.with_batch(2)
    g, w = workloads.make_inputs(wl, seed=0)
    assert dg.conv2d_grad_input_select_kernel(params(dg, wl, g, w), 1) == dg.DGRAD_KERNEL_TC_POSM
    out = run(dg, wl, g, w)
    assert rel_err(out.cpu().numpy(), full_oracle(wl, g, w)) <= TOL


def test_resnet_full_size_every_element(dg, parity_log):
    # 448 tiles on at most 152 CTAs: every CTA takes several tiles, so both
    # TMEM accumulator buffers, the ring wrap-around and the next-tile
    # prefetch run under an element-by-element check against the oracle.
    wl = workloads.RESNET
    g, w = workloads.make_inputs(wl, seed=0)
    assert dg.conv2d_grad_input_select_kernel(params(dg, wl, g, w), 1) == dg.DGRAD_KERNEL_TC_POSM
    out = run(dg, wl, g, w, via="prepacked")
    err = rel_err(out.cpu().numpy(), full_oracle(wl, g, w))
    parity_log("positions-on-M, resnet full size", err, TOL)
    assert err <= TOL


SHAPES = {
    # (N, Ci, H, W, Co, kH, kW, s, ph, pw)
    "ragged_rows": (1, 64, 13, 56, 64, 3, 3, 1, 1, 1),
    "channels_not_16": (2, 40, 9, 24, 48, 3, 3, 1, 1, 1),
    "pointwise": (2, 32, 10, 16, 64, 1, 1, 1, 0, 0),
    "two_by_two": (1, 16, 9, 15, 32, 2, 2, 1, 1, 1),
    "one_by_three": (1, 64, 6, 32, 64, 1, 3, 1, 0, 1),
    "pw0": (2, 64, 10, 18, 64, 3, 3, 1, 1, 0),
    "pw2": (1, 32, 8, 30, 32, 3, 3, 1, 1, 2),
    "single_row_image": (3, 8, 1, 8, 8, 3, 3, 1, 1, 1),
    "narrow_channels": (2, 1, 5, 8, 1, 3, 3, 1, 1, 1),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_shapes(dg, name, dtype):
    wl = case(SHAPES[name], dtype)
    g, w = workloads.make_inputs(wl, seed=sorted(SHAPES).index(name))
    code = dg.DTYPE_CODE[dtype]
    assert dg.conv2d_grad_input_select_kernel(params(dg, wl, g, w), code) == dg.DGRAD_KERNEL_TC_POSM
    out = run(dg, wl, g, w)
    assert rel_err(out.cpu().numpy(), full_oracle(wl, g, w)) <= TOL, name


def test_outside_the_mode_runs_general(dg):
    for shape, dtype in [((1, 8, 8, 9, 8, 3, 3, 1, 1, 1), "bf16"),   # 18-byte grad_out rows
                         ((1, 8, 8, 8, 8, 3, 3, 1, 1, 1), "f32"),
                         ((1, 72, 8, 8, 8, 3, 3, 1, 1, 1), "bf16"),   # Ci > 64
                         ((1, 8, 8, 8, 8, 5, 5, 1, 2, 2), "bf16")]:   # kW > 3
        wl = case(shape, dtype)
        g, w = workloads.make_inputs(wl, seed=1)
        p = params(dg, wl, g, w)
        assert dg.conv2d_grad_input_select_kernel(p, dg.DTYPE_CODE[dtype]) == dg.DGRAD_KERNEL_TC
        out = run(dg, wl, g, w)
        assert rel_err(out.cpu().numpy(), full_oracle(wl, g, w)) <= (5e-3 if dtype == "f32" else TOL)


def test_unaligned_grad_out_falls_back(dg):
    # grad_out 2 bytes past a 16-byte boundary: no TMA gather, so the launch
    # takes the general plan (same packed weights).
    wl = case((2, 64, 9, 16, 64, 3, 3, 1, 1, 1), "bf16")
    g, w = workloads.make_inputs(wl, seed=3)
    out = run(dg, wl, g, w, g_offset=1)
    assert rel_err(out.cpu().numpy(), full_oracle(wl, g, w)) <= TOL


def test_withheld_signal_times_out(dg):
    wl = workloads.RESNET.with_batch(1)
    g, w = workloads.make_inputs(wl, seed=0)
    dev = torch.device("cuda")
    gd, wd = g.to(dev), w.to(dev)
    out = torch.zeros(wl.grad_in_shape, device=dev)
    p = params(dg, wl, g, w)
    assert dg.conv2d_grad_input_check_errors() == 0
    dg.conv2d_grad_input_set_wait_limit_ns(50_000_000)
    dg.conv2d_grad_input_set_debug(dg.DGRAD_DEBUG_SKIP_ARRIVE)
    try:
        dg.conv2d_grad_input(gd, wd, out, p, dg.DGRAD_BF16)
        rc = dg.conv2d_grad_input_check_errors()
    finally:
        dg.conv2d_grad_input_set_debug(0)
        dg.conv2d_grad_input_set_wait_limit_ns(0)
    assert rc == 6, dg.conv2d_grad_input_status_string(rc)
    dg.conv2d_grad_input(gd, wd, out, p, dg.DGRAD_BF16)
    assert dg.conv2d_grad_input_check_errors() == 0
    assert rel_err(out.cpu().numpy(), full_oracle(wl, g, w)) <= TOL
