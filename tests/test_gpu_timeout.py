"""Failure detection on the GPU without a fault: a device-side wait is made to
run out (a stage signal that is withheld on purpose), the kernel returns on
its own, and the host reads the timeout status; the context stays usable."""
import pytest
import torch

import oracle
from conv2d_backward_implicit_gb300 import workloads

pytestmark = pytest.mark.gpu


def test_withheld_signal_times_out_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import conv2d_backward_implicit_gb300 as dg
    wl = workloads.RESNET.with_batch(1)
    g, w = workloads.make_inputs(wl, seed=0)
    dev = torch.device("cuda")
    gd, wd = g.to(dev), w.to(dev)
    out = torch.zeros(wl.grad_in_shape, device=dev)
    p = dg.params_from_shapes(g.shape, w.shape, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    assert dg.conv2d_grad_input_check_errors() == 0
    dg.conv2d_grad_input_set_wait_limit_ns(50_000_000)  # 50 ms
    dg.conv2d_grad_input_set_debug(dg.DGRAD_DEBUG_SKIP_ARRIVE)
    try:
        dg.conv2d_grad_input(gd, wd, out, p, dg.DGRAD_BF16)
        rc = dg.conv2d_grad_input_check_errors()
    finally:
        dg.conv2d_grad_input_set_debug(0)
        dg.conv2d_grad_input_set_wait_limit_ns(0)
    assert rc == 6, dg.conv2d_grad_input_status_string(rc)
    # The flag was cleared and the next call runs normally.
    dg.conv2d_grad_input(gd, wd, out, p, dg.DGRAD_BF16)
    assert dg.conv2d_grad_input_check_errors() == 0
    ref = oracle.dgrad(g.double().numpy(), w.double().numpy(), wl.H, wl.W, 1, 1, 1)
    got = out.cpu().double().numpy()
    assert abs(got - ref).max() / abs(ref).max() <= 2e-3
