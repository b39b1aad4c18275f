"""GPU parity at full size, every element, against the CPU oracle.

The five workloads run in the launch configuration the benchmark times (weights
packed beforehand, or packed by the kernel itself) and through the one-call
API (the two agree bit for bit); the whole grad_in tensor is compared with the
oracle's.  Then one case per kernel variant with several tiles for every CTA
of the persistent grid (more than two tiles per SM on a 152-SM GB300), so the
paths that only run from a CTA's second tile on -- the second TMEM
accumulator buffer, the wrap-around of the grad_out, raw-slice and weight
rings, the next-tile L2 prefetch -- are under an exact check too.

Bar: max|gpu - oracle| / max|oracle| <= 2e-3 (bf16 / fp16 inputs, the oracle
fed the identical rounded values) or 5e-3 (fp32 inputs on TF32 tensor cores),
over every element.  Each case's error is printed in the run's summary.
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
    yield mod
    mod.conv2d_grad_input_set_kernel(mod.DGRAD_KERNEL_AUTO)


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), "non-finite output"
    return float(np.max(np.abs(got - ref))) / max(float(np.max(np.abs(ref))), 1e-30)


_ORACLE = {}


def oracle_full(name, wl, g, w):
    """The whole grad_in from the oracle (cached per case name: several cases
    share a workload and its seeded inputs)."""
    if name not in _ORACLE:
        _ORACLE[name] = oracle.dgrad(g.double().numpy(), w.double().numpy(), wl.H, wl.W,
                                     wl.stride, wl.padding_h, wl.padding_w)
    return _ORACLE[name]


def on_device(t, offset=0):
    """t on the GPU, starting `offset` elements into a larger buffer (offset 1
    takes the pointer off every boundary wider than one element)."""
    dev = torch.device("cuda")
    if not offset:
        return t.to(dev)
    flat = torch.zeros(t.numel() + offset, dtype=t.dtype, device=dev)
    flat[offset:] = t.reshape(-1).to(dev)
    return flat[offset:].view(t.shape)


def run(dg, wl, g, w, via="prepacked", g_off=0, gi_off=0):
    dev = torch.device("cuda")
    gd, wd = on_device(g, g_off), w.to(dev)
    n = int(np.prod(wl.grad_in_shape))
    buf = torch.full((n + gi_off,), float("nan"), device=dev)
    out = buf[gi_off:].view(wl.grad_in_shape)
    p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    code = dg.DTYPE_CODE[wl.dtype]
    if via == "call":
        dg.conv2d_grad_input(gd, wd, out, p, code)
    else:
        ws = dg.conv2d_grad_input_workspace_size(p, code)
        if ws:
            packed = torch.empty(ws, dtype=torch.uint8, device=dev)
            dg.conv2d_grad_input_pack_weight(wd, packed, ws, p, code)
            dg.conv2d_grad_input_prepacked(gd, packed, out, p, code)
        else:  # the kernel packs the weights itself, or reads them unpacked
            dg.conv2d_grad_input_prepacked(gd, wd, out, p, code)
    rc = dg.conv2d_grad_input_check_errors()
    assert rc == 0, dg.conv2d_grad_input_status_string(rc)
    if gi_off:
        assert torch.isnan(buf[:gi_off]).all()  # nothing written before grad_in
    return out


@pytest.mark.parametrize("key", ["tiny", "resnet", "strided", "pointwise", "stem"])
def test_workload_full_size_every_element(dg, key, parity_log):
    wl = workloads.BY_KEY[key]
    g, w = workloads.make_inputs(wl, seed=0)
    p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    assert dg.conv2d_grad_input_select_kernel(p, dg.DTYPE_CODE[wl.dtype]) == dg.DGRAD_KERNEL_TC
    out = run(dg, wl, g, w, via="prepacked")   # the benchmark's launch path
    out2 = run(dg, wl, g, w, via="call")       # the one-call API
    assert torch.equal(out, out2)
    err = rel_err(out.cpu().numpy(), oracle_full(wl.name, wl, g, w))
    parity_log(f"{key} full size", err, TOL[wl.dtype])
    assert err <= TOL[wl.dtype], f"{wl.name}: {err:.3g}"


def _wl(name, N, Ci, H, W, Co, k, s, p, dtype):
    OH, OW = oracle.out_size(H, k, p, s), oracle.out_size(W, k, p, s)
    return workloads.Workload(name, N, Ci, H, W, Co, k, k, s, p, p, OH, OW, dtype, "normal",
                              (2.0 / (Ci * k * k)) ** 0.5)


# name: (workload, grad_out element offset, grad_in element offset), each
# with its own oracle cache key; tile counts for a 152-SM GPU.
MULTI_TILE = {
    # general mode, raw slices through a TMA map of two-row groups (120-byte
    # rows), TMA-store epilogue, weights packed by the kernel: 480 tiles
    "general_tma_60x60": (_wl("60x60", 32, 64, 60, 60, 64, 3, 1, 1, "bf16"), 0, 0),
    # grad_out off a 16-byte boundary: the general plan with the register
    # gather instead of the 64-wide frame: 448 tiles
    "general_register_gather": (workloads.RESNET, 1, 0),
    # grad_in off a 16-byte boundary: the general plan with the staged epilogue
    "general_staged_epilogue": (workloads.RESNET, 0, 1),
    # weights streamed through the weight ring (288 KB packed), pack kernel: 320 tiles
    "general_streamed_weights": (_wl("streamed", 80, 128, 28, 28, 128, 3, 1, 1, "bf16"), 0, 0),
    # kind::tf32, 32-channel stages, pack kernel: 448 tiles
    "general_tf32": (_wl("tf32", 32, 32, 56, 56, 32, 3, 1, 1, "f32"), 0, 0),
    # MN-major grad_out operand: 320 whole-image tiles
    "mn_major_160_images": (workloads.POINTWISE.with_batch(160), 0, 0),
    # paired column phases with the staged epilogue: 256 pairs
    "pair_staged_epilogue": (workloads.STRIDED, 0, 1),
    # stacked phases with the register gather: 896 tiles
    "stacked_register_gather": (workloads.STEM, 1, 0),
}


@pytest.mark.parametrize("name", list(MULTI_TILE))
def test_multi_tile_every_element(dg, name, parity_log):
    wl, g_off, gi_off = MULTI_TILE[name]
    g, w = workloads.make_inputs(wl, seed=0)
    p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    assert dg.conv2d_grad_input_select_kernel(p, dg.DTYPE_CODE[wl.dtype]) == dg.DGRAD_KERNEL_TC
    out = run(dg, wl, g, w, g_off=g_off, gi_off=gi_off)
    err = rel_err(out.cpu().numpy(), oracle_full(wl.name, wl, g, w))
    parity_log(f"{name} ({wl.name})", err, TOL[wl.dtype])
    assert err <= TOL[wl.dtype], f"{name}: {err:.3g}"
