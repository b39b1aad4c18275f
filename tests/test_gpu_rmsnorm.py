"""GPU parity of the fused RMSNorm + matmul (include/rmsnorm_matmul.h) with the
CPU oracle (oracle/rmsnorm_matmul_oracle.c), through the C ABI.

Inputs are drawn in float32, rounded to the input type, and the oracle gets
exactly those values (float64).  The bar is an element-wise bound from the
arithmetic, not a loose relative tolerance:
  * tensor-core kernel (bf16 / fp16): each X[i, t] * W_norm[t] is rounded to
    the input type (relative error <= u, u = 2^-8 for bf16, 2^-11 for fp16)
    before an exact product with W_proj and float32 accumulation, and r[i] is
    applied in float32, so
        |C - C_exact| <= r[i] * (u + K 2^-23) * S[i, j] + 2^-20 |C_exact|,
    S = (|X| |W_norm|) |W_proj| (the sum of the terms' magnitudes);
  * CUDA-core kernel (every dtype, float32 arithmetic throughout):
        |C - C_exact| <= r[i] * K 2^-22 * S[i, j] + 2^-20 |C_exact|.
Each case also prints max|C - C_exact| / max|C_exact| in the run's summary.
"""
import numpy as np
import pytest
import torch

from oracle import rmsnorm as orn

pytestmark = pytest.mark.gpu

U = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11, "f32": 0.0}
TORCH = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module")
def dg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import conv2d_backward_implicit_gb300 as mod
    mod.library()
    yield mod
    mod.rmsnorm_matmul_set_kernel(mod.DGRAD_KERNEL_AUTO)


def make_inputs(m, n, k, dtype, seed):
    """X ~ N(0, 1) rows with per-row scales over two decades, W_norm ~ U(0.5, 1.5),
    W_proj ~ N(0, 1/k): rounded to the input type."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(m, k, generator=g) * torch.exp(torch.empty(m, 1).uniform_(-2.3, 2.3, generator=g))
    wn = torch.empty(k).uniform_(0.5, 1.5, generator=g)
    wp = torch.randn(k, n, generator=g) / np.sqrt(k)
    t = TORCH[dtype]
    return x.to(t), wn.to(t), wp.to(t)


def run(dg, x, wn, wp, eps, dtype, c_offset=0):
    m, k = x.shape
    n = wp.shape[1]
    dev = torch.device("cuda")
    buf = torch.full((m * n + c_offset,), float("nan"), device=dev)
    c = buf[c_offset:].view(m, n)
    p = dg.RmsParams(m, n, k, eps)
    dg.rmsnorm_matmul(x.to(dev), wn.to(dev), wp.to(dev), c, p, dg.DTYPE_CODE[dtype])
    rc = dg.rmsnorm_matmul_check_errors()
    assert rc == 0, dg.STATUS.get(rc, rc)
    if c_offset:
        assert torch.isnan(buf[:c_offset]).all()
    return c.cpu().double().numpy()


def check(got, x, wn, wp, eps, dtype, kernel, rows=None):
    xd, wnd, wpd = x.double().numpy(), wn.double().numpy(), wp.double().numpy()
    if rows is not None:
        xd, got = xd[rows], got[rows]
    ref = orn.rmsnorm_matmul(xd, wnd, wpd, eps)
    r = orn.rms_rows(xd, eps)
    k = xd.shape[1]
    s = (np.abs(xd) * np.abs(wnd)[None, :]) @ np.abs(wpd)
    rel = (U[dtype] + k * 2.0 ** -23) if kernel == "tc" else k * 2.0 ** -22
    bound = r[:, None] * rel * s + 2.0 ** -20 * np.abs(ref)
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    worst = float(np.max(err - bound))
    assert worst <= 0, f"error above the bound by {worst:.3g} (max err {err.max():.3g})"
    return float(err.max() / max(np.abs(ref).max(), 1e-30))


# (m, n, k): one tile; ragged rows and a ragged last K stage; several tiles
# per CTA on a 152-SM GPU (256 tiles), so the second TMEM buffer, the row-scale
# buffers and the stage ring's wrap-around run; N of one tile.
TC_CASES = [(128, 256, 64), (300, 320, 520), (4096, 2048, 256), (1, 64, 8), (777, 64, 1000)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("case", TC_CASES)
def test_tensor_core_kernel(dg, dtype, case, parity_log):
    m, n, k = case
    x, wn, wp = make_inputs(m, n, k, dtype, seed=m + n + k)
    dev = torch.device("cuda")
    c = torch.empty(m, n, device=dev)
    p = dg.RmsParams(m, n, k, 1e-5)
    assert dg.rmsnorm_matmul_select_kernel(x.to(dev), wn.to(dev), wp.to(dev), c, p,
                                           dg.DTYPE_CODE[dtype]) == dg.DGRAD_KERNEL_TC
    got = run(dg, x, wn, wp, 1e-5, dtype)
    err = check(got, x, wn, wp, 1e-5, dtype, "tc")
    parity_log(f"rmsnorm_matmul tc {dtype} {m}x{n}x{k}", err, U[dtype])


SIMT_CASES = [("f32", (300, 320, 520)), ("f32", (65, 70, 33)), ("bf16", (65, 70, 33)),
              ("f16", (130, 100, 9)), ("bf16", (300, 320, 520))]


@pytest.mark.parametrize("dtype,case", SIMT_CASES)
def test_cuda_core_kernel(dg, dtype, case, parity_log):
    m, n, k = case
    x, wn, wp = make_inputs(m, n, k, dtype, seed=7 * m + n + k)
    forced = dtype != "f32" and n % 64 == 0 and k % 8 == 0
    if forced:
        dg.rmsnorm_matmul_set_kernel(dg.DGRAD_KERNEL_SIMT)
    try:
        got = run(dg, x, wn, wp, 0.25, dtype)
    finally:
        dg.rmsnorm_matmul_set_kernel(dg.DGRAD_KERNEL_AUTO)
    err = check(got, x, wn, wp, 0.25, dtype, "simt")
    parity_log(f"rmsnorm_matmul simt {dtype} {m}x{n}x{k}", err, 1e-5)


def test_unaligned_output_takes_the_cuda_core_kernel(dg):
    x, wn, wp = make_inputs(128, 256, 64, "bf16", seed=3)
    got = run(dg, x, wn, wp, 1e-5, "bf16", c_offset=1)  # C off a 16-byte boundary
    check(got, x, wn, wp, 1e-5, "bf16", "simt")


def test_forced_tensor_core_kernel_refuses_an_odd_shape(dg):
    x, wn, wp = make_inputs(64, 70, 32, "bf16", seed=4)
    dg.rmsnorm_matmul_set_kernel(dg.DGRAD_KERNEL_TC)
    try:
        with pytest.raises(dg.DgradError) as e:
            run(dg, x, wn, wp, 1e-5, "bf16")
        assert e.value.status == 4  # DGRAD_ERR_UNSUPPORTED
    finally:
        dg.rmsnorm_matmul_set_kernel(dg.DGRAD_KERNEL_AUTO)


def test_full_size_sampled_rows(dg, parity_log):
    """The benchmark's workload (M = 8192 tokens, K = 4096, N = 4096, bf16) in
    one launch; the oracle checks 64 random rows plus the first and last."""
    m, n, k = 8192, 4096, 4096
    x, wn, wp = make_inputs(m, n, k, "bf16", seed=11)
    got = run(dg, x, wn, wp, 1e-6, "bf16")
    rows = np.unique(np.concatenate([[0, m - 1], np.random.default_rng(5).choice(m, 64, replace=False)]))
    err = check(got, x, wn, wp, 1e-6, "bf16", "tc", rows=rows)
    parity_log("rmsnorm_matmul tc bf16 8192x4096x4096 (66 rows)", err, U["bf16"])


def test_row_scale_invariance_on_the_gpu(dg):
    """RmsNorm makes each row of C independent of the row's scale (eps = 0):
    X and 8 X (exact in bf16) give the same C up to the kernel's rounding."""
    x, wn, wp = make_inputs(256, 512, 512, "bf16", seed=6)
    a = run(dg, x, wn, wp, 0.0, "bf16")
    b = run(dg, (x.float() * 8).to(torch.bfloat16), wn, wp, 0.0, "bf16")
    assert np.allclose(a, b, rtol=1e-5, atol=1e-6)
