"""GPU parity for the raw-slice gather's load modes and whole-row tiles.

The tensor-core kernel stages grad_out rows in shared memory before turning
them into the frame window; how a slice is loaded depends on the shape:

* tiled, one grad_out row per map row (rows a multiple of 16 bytes);
* tiled over groups of g rows (rows not a multiple of 16 bytes, planes split
  into whole g-row groups: a 28-column bf16 row needs g = 2);
* one 1-D bulk copy per channel (the g-row group is wider than a TMA box);
* one 1-D bulk copy of whole channel planes (tiles that cover whole images);
* 1x1 problems whose tiles are whole images: the grad_out operand is read
  MN-major (channel rows of positions), regrouped in 16-byte pieces;
* few input channels and stride > 1: positions on M, every phase's channels
  stacked on N, window taps as shifted views of one frame;
* stride 2 with one 128-row channel tile: the two column phases of the same
  rows are taken as a pair -- one shared window, two accumulators -- and
  stored as whole grad_in rows.

Each case below is chosen (and commented) for the mode it exercises, with
several images whose last row tile runs past the image, channel counts that
leave ragged or empty slices, strides 1 and 2 (the sub-pixel phases), and
resident or streamed weights.  Every output element is compared with the
oracle, and two launches must agree bit for bit.
"""
import numpy as np
import pytest
import torch

from conv2d_backward_implicit_gb300 import workloads

from test_gpu_parity import TOL, make_case, oracle_full, rel_err, run_gpu

pytestmark = pytest.mark.gpu

# (N, Ci, H, W, Co, kH, kW, s, ph, pw), dtype, what it exercises
CASES = [
    ((2, 64, 32, 32, 96, 3, 3, 2, 1, 1), "bf16",
     "tiled, 1 row per map row; s=2 phases; last row tile past the image; 64+32 channel chunks"),
    ((3, 72, 20, 28, 130, 3, 3, 1, 1, 1), "bf16",
     "tiled over 2-row groups (56-byte rows); 3 images; slices past Co=130"),
    ((2, 40, 36, 36, 24, 5, 5, 2, 2, 2), "f32",
     "tiled over 2-row groups, TF32; 5x5 s=2 (phases of 3x3, 3x2, 2x3, 2x2 taps); Co=24"),
    ((3, 40, 28, 28, 80, 3, 3, 2, 1, 1), "bf16",
     "whole planes (14x14 bf16 planes are not 16-byte multiples); s=2"),
    ((3, 48, 14, 14, 200, 1, 1, 1, 0, 0), "f16",
     "whole planes, 1x1 (a plain GEMM per image); Co=200 ragged"),
    ((2, 96, 20, 20, 300, 2, 2, 2, 0, 0), "bf16",
     "whole planes; even kernel s=2 (one tap per phase); five channel chunks, streamed weights"),
    ((2, 40, 24, 300, 40, 3, 3, 2, 1, 1), "bf16",
     "one 1-D copy per channel (a 4-row group of 150 columns exceeds a TMA box)"),
    ((3, 64, 24, 24, 136, 3, 3, 1, 1, 1), "f32",
     "tiled, TF32; rows per tile do not divide H; Co=136 ragged"),
    ((3, 200, 12, 12, 300, 1, 1, 1, 0, 0), "bf16",
     "MN-major grad_out operand from whole-plane copies (1x1); Co=300 leaves a 44-channel chunk"),
    ((2, 130, 16, 16, 520, 1, 1, 1, 0, 0), "f16",
     "MN-major operand from whole-plane tensor-map boxes; Ci=130: a 2-channel second tile"),
    ((2, 3, 30, 26, 24, 7, 7, 2, 3, 3), "f32",
     "stacked phases (Ci=3, s=2, 7x7: 4 x 4 window taps), 8 frame rows per tile, partial last tile"),
    ((2, 2, 25, 23, 40, 5, 3, 3, 2, 1), "bf16",
     "stacked phases, s=3: 9 phases x 2 channels on 32 columns; odd sizes; Co=40 ragged"),
    ((3, 1, 17, 40, 70, 4, 4, 4, 1, 2), "f16",
     "stacked phases, s=4: 16 phases x 1 channel; rows not a multiple of the stride; Co=70"),
    ((2, 8, 16, 16, 48, 3, 3, 2, 1, 1), "f32",
     "stacked phases, 4 phases x 8 channels = 32 columns, TF32"),
    ((2, 128, 24, 32, 72, 3, 3, 2, 1, 1), "bf16",
     "paired column phases (s=2, 128 channels): rows of W=32 from two 16-column phases"),
    ((3, 128, 20, 48, 70, 3, 3, 2, 1, 1), "f32",
     "paired column phases, TF32, W=48, Co=70 ragged"),
    ((2, 100, 16, 40, 64, 3, 3, 2, 1, 1), "bf16",
     "paired column phases, Ci=100 of a 128-row tile, W=40"),
    ((2, 100, 16, 24, 64, 5, 5, 2, 2, 2), "bf16",
     "5x5 at stride 2: the column phases read different frames, so tiles stay unpaired"),
]


@pytest.fixture(scope="module")
def dg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import conv2d_backward_implicit_gb300 as mod
    mod.library()
    return mod


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_raw_mode_case(dg, idx):
    shape, dtype, what = CASES[idx]
    wl = make_case(shape, dtype, idx)
    g, w = workloads.make_inputs(wl, seed=100 + idx)
    p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    assert dg.conv2d_grad_input_select_kernel(p, dg.DTYPE_CODE[dtype]) == dg.DGRAD_KERNEL_TC
    ref = oracle_full(wl, g, w)
    out1 = run_gpu(dg, wl, g, w).cpu().numpy()
    err = rel_err(out1, ref)
    assert err <= TOL[dtype], f"{what}: {err:.3g}"
    out2 = run_gpu(dg, wl, g, w, via="prepacked").cpu().numpy()
    assert np.array_equal(out1, out2), f"{what}: prepacked launch differs from the one-call API"


def run_offset(dg, wl, g, w, g_offset, out_offset):
    """The one-call API with grad_out / grad_in starting g_offset / out_offset
    elements past a 16-byte boundary (aligned to the element size only)."""
    dev = torch.device("cuda")
    flat = torch.zeros(g.numel() + g_offset, dtype=g.dtype, device=dev)
    flat[g_offset:] = g.reshape(-1).to(dev)
    gd = flat[g_offset:].view(g.shape)
    n_out = int(np.prod(wl.grad_in_shape))
    oflat = torch.full((n_out + out_offset,), float("nan"), device=dev)
    out = oflat[out_offset:].view(wl.grad_in_shape)
    p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    dg.conv2d_grad_input(gd, w.to(dev), out, p, dg.DTYPE_CODE[wl.dtype])
    assert dg.conv2d_grad_input_check_errors() == 0
    return out.cpu().numpy()


# One case of each mode whose plan needs aligned pointers for its TMA / bulk
# copies: the MN-major 1x1 operand, the stacked phases and the paired column
# phases.  A misaligned grad_out (no raw-slice copies) or grad_in (no TMA
# stores) must take the mode's fallback and still match the oracle.
ALIGN_CASES = [8, 10, 14]


@pytest.mark.parametrize("idx", ALIGN_CASES)
@pytest.mark.parametrize("g_offset,out_offset", [(1, 0), (0, 1), (3, 5)])
def test_mode_pointer_fallbacks(dg, idx, g_offset, out_offset):
    shape, dtype, what = CASES[idx]
    wl = make_case(shape, dtype, idx)
    g, w = workloads.make_inputs(wl, seed=300 + idx)
    got = run_offset(dg, wl, g, w, g_offset, out_offset)
    err = rel_err(got, oracle_full(wl, g, w))
    assert err <= TOL[dtype], f"{what}, offsets {g_offset}/{out_offset}: {err:.3g}"
