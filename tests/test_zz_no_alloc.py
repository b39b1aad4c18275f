"""conv2d_grad_input_noalloc: the allocation-free entry point for callers that
cannot allocate device memory (graph captures that forbid allocation, runtimes
whose arena owns the device, latency-critical loops).  It must give the same
result as the allocating conv2d_grad_input, call after call, even though every
call reuses the same fixed scratch array left over from the previous one.

Collected last on purpose, so that a run stopping at its first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from conv2d_backward_implicit_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-3, "f16": 2e-3, "f32": 5e-3}


def _rel_err(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    assert np.isfinite(a).all()
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


def test_noalloc_matches_allocating_entry_point_twice_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import conv2d_backward_implicit_gb300 as dg
    dev = torch.device("cuda")
    # Two different problems back to back: the second call finds the first
    # call's packed weights (a larger pack) still in the shared scratch array.
    cases = [workloads.STRIDED.with_batch(2), workloads.RESNET.with_batch(2),
             workloads.STEM.with_batch(1)]
    for wl in cases:
        g, w = workloads.make_inputs(wl, seed=7)
        gd, wd = g.to(dev), w.to(dev)
        p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h,
                                  wl.padding_w)
        code = dg.DTYPE_CODE[wl.dtype]
        assert dg.conv2d_grad_input_select_kernel(p, code) == dg.DGRAD_KERNEL_TC
        ref = torch.full(wl.grad_in_shape, float("nan"), device=dev)
        dg.conv2d_grad_input(gd, wd, ref, p, code)
        for _ in range(2):
            out = torch.full(wl.grad_in_shape, float("nan"), device=dev)
            dg.conv2d_grad_input_noalloc(gd, wd, out, p, code)
            assert dg.conv2d_grad_input_check_errors() == 0
            assert _rel_err(out, ref) <= TOL[wl.dtype], wl.name


def test_noalloc_rejects_packs_above_its_limit():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import conv2d_backward_implicit_gb300 as dg
    # 1024 x 1024 x 3x3 bf16 weights pack to 18.9 MB > 8 MiB.
    p = dg.Params(1, 1024, 8, 8, 1024, 3, 3, 1, 1, 8, 8, 1)
    assert dg.conv2d_grad_input_workspace_size(p, dg.DGRAD_BF16) > 8 * 2**20
    g = torch.zeros((1, 1024, 8, 8), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((1024, 1024, 3, 3), dtype=torch.bfloat16, device="cuda")
    out = torch.full((1, 1024, 8, 8), 3.0, device="cuda")
    with pytest.raises(dg.DgradError) as ei:
        dg.conv2d_grad_input_noalloc(g, w, out, p, dg.DGRAD_BF16)
    assert ei.value.status == 7
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)


def _pool_high_water():
    """Read and reset functions for the used-memory high-water mark of the
    current device's memory pool -- the pool cudaMallocAsync draws from (driver
    API, so no particular CUDA runtime copy is involved)."""
    cu = ctypes.CDLL("libcuda.so.1")
    dev = ctypes.c_int()
    assert cu.cuCtxGetDevice(ctypes.byref(dev)) == 0
    pool = ctypes.c_void_p()
    assert cu.cuDeviceGetMemPool(ctypes.byref(pool), dev) == 0
    used_mem_high = 8  # CU_MEMPOOL_ATTR_USED_MEM_HIGH

    def high():
        v = ctypes.c_uint64()
        assert cu.cuMemPoolGetAttribute(pool, used_mem_high, ctypes.byref(v)) == 0
        return v.value

    def reset():
        z = ctypes.c_uint64(0)  # resets the mark to the memory in use now
        assert cu.cuMemPoolSetAttribute(pool, used_mem_high, ctypes.byref(z)) == 0

    return high, reset


def test_noalloc_takes_no_device_memory_after_its_first_call():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import conv2d_backward_implicit_gb300 as dg
    dev = torch.device("cuda")
    high, reset = _pool_high_water()
    for wl in (workloads.STRIDED.with_batch(1), workloads.STEM.with_batch(1)):
        g, w = workloads.make_inputs(wl, seed=3)
        gd, wd = g.to(dev), w.to(dev)
        p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h,
                                  wl.padding_w)
        code = dg.DTYPE_CODE[wl.dtype]
        ws = dg.conv2d_grad_input_workspace_size(p, code)
        assert ws > 0  # a layer whose weights are packed into scratch memory
        out = torch.empty(wl.grad_in_shape, device=dev)
        dg.conv2d_grad_input_noalloc(gd, wd, out, p, code)  # first call: address set-up
        torch.cuda.synchronize()
        # The probe sees the allocating entry point's stream-ordered workspace ...
        reset()
        before = high()
        dg.conv2d_grad_input(gd, wd, out, p, code)
        torch.cuda.synchronize()
        assert high() >= before + ws, wl.name
        # ... and nothing from the allocation-free one.
        reset()
        before = high()
        for _ in range(3):
            dg.conv2d_grad_input_noalloc(gd, wd, out, p, code)
        torch.cuda.synchronize()
        assert high() == before, wl.name
        assert dg.conv2d_grad_input_check_errors() == 0
