"""GPU parity of the general tensor-core mode on the 64-wide frame (stride 1,
bf16 / fp16, rows of at most 56 columns, resident packed weights) against the
CPU oracle: shapes across that range (grad_out rows a multiple of 16 bytes,
W a multiple of 4) -- ragged row tiles, channel counts that are not multiples
of 16, one and two 128-row input-channel tiles, several 64-channel grad_out
chunks, 1x1 to 3x3 kernels, paddings 0..2 -- and the
fallback to the Wr + Jw - 1 frame when grad_out or grad_in is not 16-byte
aligned.  The kernel packs these layers' weights in shared memory itself
(workspace size 0): with 16-byte vector loads when the weight rows allow it,
else with scalar loads, and both give the same bits.
Bar: max|gpu - oracle| / max|oracle| <= 2e-3."""
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
    mod.conv2d_grad_input_set_kernel(mod.DGRAD_KERNEL_AUTO)
    return mod


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


def run(dg, wl, g, w, g_offset=0, out_offset=0, w_offset=0):
    dev = torch.device("cuda")
    flat = torch.zeros(g.numel() + g_offset, dtype=g.dtype, device=dev)
    flat[g_offset:] = g.reshape(-1).to(dev)
    gd = flat[g_offset:].view(g.shape)
    wflat = torch.zeros(w.numel() + w_offset, dtype=w.dtype, device=dev)
    wflat[w_offset:] = w.reshape(-1).to(dev)
    wd = wflat[w_offset:].view(w.shape)
    n_out = int(np.prod(wl.grad_in_shape))
    oflat = torch.full((n_out + out_offset,), float("nan"), device=dev)
    out = oflat[out_offset:].view(wl.grad_in_shape)
    p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    dg.conv2d_grad_input(gd, wd, out, p, dg.DTYPE_CODE[wl.dtype])
    rc = dg.conv2d_grad_input_check_errors()
    assert rc == 0, dg.conv2d_grad_input_status_string(rc)
    return out


def oracle_of(wl, g, w):
    return oracle.dgrad(g.double().numpy(), w.double().numpy(), wl.H, wl.W, wl.stride,
                        wl.padding_h, wl.padding_w)


SHAPES = {
    # (N, Ci, H, W, Co, kH, kW, s, ph, pw)
    "resnet_rows_ragged": (1, 64, 13, 56, 64, 3, 3, 1, 1, 1),
    "channels_not_16": (2, 40, 9, 24, 48, 3, 3, 1, 1, 1),
    "pointwise_two_chunks_m128": (2, 128, 8, 16, 128, 1, 1, 1, 0, 0),
    "pointwise_two_m_tiles": (2, 200, 5, 8, 40, 1, 1, 1, 0, 0),
    "pointwise_ragged_chunks": (1, 100, 6, 24, 72, 1, 1, 1, 0, 0),
    "one_by_three": (1, 64, 6, 32, 64, 1, 3, 1, 0, 1),
    "three_by_one": (1, 32, 10, 16, 48, 3, 1, 1, 1, 0),
    "pad2_1x1": (1, 16, 6, 12, 16, 1, 1, 1, 2, 2),
    "pad0_3x1": (2, 16, 10, 16, 24, 3, 1, 1, 0, 0),
    "single_row_image": (3, 8, 1, 8, 8, 3, 3, 1, 1, 1),
    "narrow_channels": (2, 1, 5, 8, 1, 3, 3, 1, 1, 1),
    "wide_56_pad0_1x1": (1, 16, 3, 56, 16, 1, 1, 1, 0, 0),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_shapes(dg, name, dtype):
    wl = case(SHAPES[name], dtype)
    g, w = workloads.make_inputs(wl, seed=sorted(SHAPES).index(name))
    out = run(dg, wl, g, w)
    assert rel_err(out.cpu().numpy(), oracle_of(wl, g, w)) <= TOL, name


@pytest.mark.parametrize("g_offset,out_offset", [(1, 0), (0, 1), (8, 4)])
def test_pointer_alignment_fallback(dg, g_offset, out_offset):
    # grad_out 2 bytes, or grad_in 4 bytes, past a 16-byte boundary: the launch
    # takes the plan on the Wr + Jw - 1 frame; 16-byte offsets keep this one.
    wl = case((2, 64, 9, 16, 64, 3, 3, 1, 1, 1), "bf16")
    g, w = workloads.make_inputs(wl, seed=3)
    out = run(dg, wl, g, w, g_offset=g_offset, out_offset=out_offset)
    assert rel_err(out.cpu().numpy(), oracle_of(wl, g, w)) <= TOL


@pytest.mark.parametrize("name", ["resnet_rows_ragged", "channels_not_16", "pointwise_two_m_tiles"])
def test_in_kernel_pack_vector_and_scalar_loads_agree(dg, name):
    # A weight pointer 16 bytes past a boundary keeps the vector loads; 2 bytes
    # past one takes the scalar loads.  Both write the same packed image, so
    # grad_in matches bit for bit (and the oracle within the bar).
    wl = case(SHAPES[name], "bf16")
    g, w = workloads.make_inputs(wl, seed=7)
    p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    assert dg.conv2d_grad_input_workspace_size(p, dg.DGRAD_BF16) == 0
    ref = run(dg, wl, g, w).cpu().numpy()
    assert rel_err(ref, oracle_of(wl, g, w)) <= TOL
    for w_offset in (8, 1):
        out = run(dg, wl, g, w, w_offset=w_offset).cpu().numpy()
        assert np.array_equal(out, ref), (name, w_offset)


def test_in_kernel_pack_with_the_alignment_fallback(dg):
    # grad_out off a 16-byte boundary: the general plan on the Wr + Jw - 1 frame
    # runs, and it too packs the weights in the kernel (scalar loads here).
    wl = case((2, 64, 9, 16, 64, 3, 3, 1, 1, 1), "f16")
    g, w = workloads.make_inputs(wl, seed=9)
    out = run(dg, wl, g, w, g_offset=1, w_offset=3)
    assert rel_err(out.cpu().numpy(), oracle_of(wl, g, w)) <= TOL


def test_prepacked_takes_the_weights_when_nothing_is_packed(dg):
    wl = case(SHAPES["resnet_rows_ragged"], "bf16")
    g, w = workloads.make_inputs(wl, seed=11)
    dev = torch.device("cuda")
    p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    assert dg.conv2d_grad_input_workspace_size(p, dg.DGRAD_BF16) == 0
    gd, wd = g.to(dev), w.to(dev)
    buf = torch.full((64,), 7, dtype=torch.uint8, device=dev)
    dg.conv2d_grad_input_pack_weight(wd, buf, 0, p, dg.DGRAD_BF16)  # nothing to pack
    out = torch.full(wl.grad_in_shape, float("nan"), device=dev)
    dg.conv2d_grad_input_prepacked(gd, wd, out, p, dg.DGRAD_BF16)
    assert dg.conv2d_grad_input_check_errors() == 0
    torch.cuda.synchronize()
    assert torch.all(buf == 7)
    ref = run(dg, wl, g, w)
    assert torch.equal(out, ref)
