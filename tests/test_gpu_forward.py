"""GPU parity for the forward convolution entry point (conv2d_forward).

At stride 1 the forward convolution of a layer is the input gradient of the
layer with the channel axes swapped, the kernel flipped and padding
kernel - 1 - padding; conv2d_forward runs it through the same kernels.  At
stride s > 1 it is one stride-1 valid correlation of a space-to-depth copy of
x with rearranged weights (the identity is checked on the CPU in
test_forward_decomposition_cpu.py), run the same way.  It is
checked element by element against the oracle's own forward convolution
(a direct loop over outputs, pinned independently of the dgrad oracle), and
the adjoint identity <conv(x), g> = <x, dgrad(g)> is checked with both sides
computed on the GPU.
"""
import numpy as np
import pytest
import torch

import oracle
from conv2d_backward_implicit_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-3, "f16": 2e-3, "f32": 5e-3}


@pytest.fixture(scope="module")
def dg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import conv2d_backward_implicit_gb300 as mod
    mod.library()
    return mod


def layer(shape, dtype, s=1):
    N, Ci, H, W, Co, kH, kW, ph, pw = shape
    OH, OW = oracle.out_size(H, kH, ph, s), oracle.out_size(W, kW, pw, s)
    return workloads.Workload(f"layer{shape}", N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW, dtype,
                              "uniform")


def forward_gpu(dg, wl, x, w):
    dev = torch.device("cuda")
    out = torch.full((wl.N, wl.Co, wl.OH, wl.OW), float("nan"), device=dev, dtype=torch.float32)
    p = dg.params_from_shapes((wl.N, wl.Co, wl.OH, wl.OW), w.shape, wl.H, wl.W, wl.stride,
                              wl.padding_h, wl.padding_w)
    dg.conv2d_forward(x.to(dev), w.to(dev), out, p, dg.DTYPE_CODE[wl.dtype])
    assert dg.conv2d_grad_input_check_errors() == 0
    return out.cpu().double().numpy()


def dgrad_gpu(dg, wl, g, w):
    dev = torch.device("cuda")
    out = torch.full(wl.grad_in_shape, float("nan"), device=dev, dtype=torch.float32)
    p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    dg.conv2d_grad_input(g.to(dev), w.to(dev), out, p, dg.DTYPE_CODE[wl.dtype])
    assert dg.conv2d_grad_input_check_errors() == 0
    return out.cpu().double().numpy()


def inputs(wl, seed):
    """x [N,Ci,H,W] and weight [Co,Ci,kH,kW], U[-1,1], rounded to the dtype."""
    gen = torch.Generator().manual_seed(seed)
    x = (torch.rand((wl.N, wl.Ci, wl.H, wl.W), generator=gen) * 2 - 1).to(workloads.TORCH_DTYPE[wl.dtype])
    w = (torch.rand(wl.weight_shape, generator=gen) * 2 - 1).to(workloads.TORCH_DTYPE[wl.dtype])
    return x, w


SHAPES = {
    # (N, Ci, H, W, Co, kH, kW, ph, pw)
    "resnet_like_3x3": (2, 64, 14, 14, 64, 3, 3, 1, 1),
    "pointwise": (2, 96, 9, 11, 160, 1, 1, 0, 0),
    "rect_kernel_ph_ne_pw": (2, 12, 11, 15, 20, 5, 3, 2, 0),
    "even_kernel_p0": (3, 8, 9, 9, 8, 2, 2, 0, 0),
    "even_kernel_p1": (1, 16, 10, 7, 24, 2, 2, 1, 1),
    "stem_like_7x7": (2, 3, 20, 18, 24, 7, 7, 3, 3),
    "co_ragged": (2, 40, 12, 16, 70, 3, 3, 0, 1),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_forward_matches_oracle(dg, name, dtype):
    wl = layer(SHAPES[name], dtype)
    x, w = inputs(wl, sorted(SHAPES).index(name))
    got = forward_gpu(dg, wl, x, w)
    ref = oracle.conv2d_forward(x.double().numpy(), w.double().numpy(), 1, wl.padding_h, wl.padding_w)
    assert got.shape == ref.shape
    assert np.isfinite(got).all()
    err = float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))
    assert err <= TOL[dtype], f"{name}: {err:.3g}"


@pytest.mark.parametrize("name", ["resnet_like_3x3", "rect_kernel_ph_ne_pw", "stem_like_7x7"])
def test_adjoint_identity_on_gpu(dg, name):
    # <conv(x), g> = <x, dgrad(g)>, each side from the GPU; the bound is the
    # tolerance times the sums of absolute products on each side.
    wl = layer(SHAPES[name], "bf16")
    x, w = inputs(wl, 7)
    gen = torch.Generator().manual_seed(8)
    g = (torch.rand((wl.N, wl.Co, wl.OH, wl.OW), generator=gen) * 2 - 1).to(torch.bfloat16)
    y = forward_gpu(dg, wl, x, w)
    gi = dgrad_gpu(dg, wl, g, w)
    xd, gd = x.double().numpy(), g.double().numpy()
    lhs, rhs = float(np.sum(y * gd)), float(np.sum(xd * gi))
    scale = float(np.sum(np.abs(y * gd)) + np.sum(np.abs(xd * gi)))
    assert abs(lhs - rhs) <= 2e-3 * scale, (lhs, rhs, scale)


STRIDED = {
    # (N, Ci, H, W, Co, kH, kW, ph, pw), stride
    "downsample_3x3_s2": ((2, 32, 16, 16, 64, 3, 3, 1, 1), 2),
    "downsample_1x1_s2": ((2, 64, 14, 14, 128, 1, 1, 0, 0), 2),
    "stem_7x7_s2": ((2, 3, 30, 26, 24, 7, 7, 3, 3), 2),
    "rect_3x2_s3_ph_ne_pw": ((1, 12, 17, 13, 20, 3, 2, 2, 0), 3),
    "k2_s4": ((2, 8, 19, 17, 8, 2, 2, 1, 0), 4),
    "odd_sizes_5x3_s2": ((2, 10, 13, 11, 14, 5, 3, 0, 2), 2),
    "padding_at_kernel_1x1_s3": ((1, 6, 8, 9, 5, 1, 1, 1, 1), 3),
}


@pytest.mark.parametrize("name", sorted(STRIDED))
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_strided_forward_matches_oracle(dg, name, dtype):
    shape, s = STRIDED[name]
    wl = layer(shape, dtype, s)
    x, w = inputs(wl, 100 + sorted(STRIDED).index(name))
    got = forward_gpu(dg, wl, x, w)
    ref = oracle.conv2d_forward(x.double().numpy(), w.double().numpy(), s, wl.padding_h, wl.padding_w)
    assert got.shape == ref.shape
    assert np.isfinite(got).all()
    err = float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))
    assert err <= TOL[dtype], f"{name} {dtype}: {err:.3g}"


def test_strided_forward_full_size_layer(dg, parity_log):
    # The strided workload's layer (56x56 -> 28x28, 128 -> 256 channels, 3x3
    # s2 p1), forward, every element against the oracle.
    wl = layer((32, 128, 56, 56, 256, 3, 3, 1, 1), "bf16", 2)
    x, w = inputs(wl, 3)
    got = forward_gpu(dg, wl, x, w)
    ref = oracle.conv2d_forward(x.double().numpy(), w.double().numpy(), 2, 1, 1)
    err = float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))
    parity_log("forward, strided 3x3 s2 layer full size", err, TOL["bf16"])
    assert err <= TOL["bf16"]


@pytest.mark.parametrize("name", ["downsample_3x3_s2", "stem_7x7_s2", "rect_3x2_s3_ph_ne_pw"])
def test_strided_adjoint_identity_on_gpu(dg, name):
    # <conv(x), g> = <x, dgrad(g)> at stride > 1, each side from the GPU.
    shape, s = STRIDED[name]
    wl = layer(shape, "bf16", s)
    x, w = inputs(wl, 9)
    gen = torch.Generator().manual_seed(10)
    g = (torch.rand((wl.N, wl.Co, wl.OH, wl.OW), generator=gen) * 2 - 1).to(torch.bfloat16)
    y = forward_gpu(dg, wl, x, w)
    gi = dgrad_gpu(dg, wl, g, w)
    xd, gd = x.double().numpy(), g.double().numpy()
    lhs, rhs = float(np.sum(y * gd)), float(np.sum(xd * gi))
    scale = float(np.sum(np.abs(y * gd)) + np.sum(np.abs(xd * gi)))
    assert abs(lhs - rhs) <= 2e-3 * scale, (lhs, rhs, scale)
