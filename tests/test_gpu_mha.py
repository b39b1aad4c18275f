"""GPU parity of the attention dV (include/mha_grad_v.h) with the CPU oracle
(oracle/mha_grad_v_oracle.c), through the C ABI.

Q, K and dO are drawn in float32 and rounded to the input type; the oracle
gets those values (float64) and makes the LSE input from them (the forward
statistics over the keys each query attends), which both sides then read.
The bar is element-wise: dV is linear in dO with P >= 0, so A = the oracle's
dV for |dO| is the sum of the terms' magnitudes, and
  |dV - dV_exact| <= c * A + 1e-6 * max|dV_exact|,
c = 1e-4 for the CUDA-core kernel (float32 scores, exp and sums) and
2^-8 + 1e-4 (bf16) or 2^-11 + 1e-4 (fp16) for the tensor-core kernel, which
also rounds P to the input type for its second product.
"""
import numpy as np
import pytest
import torch

from oracle import mha

pytestmark = pytest.mark.gpu

TORCH = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
C_TC = {"bf16": 2.0 ** -8 + 1e-4, "f16": 2.0 ** -11 + 1e-4}


@pytest.fixture(scope="module")
def dg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import conv2d_backward_implicit_gb300 as mod
    mod.library()
    yield mod
    mod.mha_grad_v_set_kernel(mod.DGRAD_KERNEL_AUTO)


def make_inputs(q_seq, kv_seq, nh, nkv, hd, window, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    kv = mha.kv_len(q_seq, kv_seq)
    t = TORCH[dtype]
    q = torch.randn(q_seq, nh, hd, generator=g).to(t)
    k = torch.randn(kv, nkv, hd, generator=g).to(t)
    go = torch.randn(q_seq, nh, hd, generator=g).to(t)
    lse = mha.forward_lse(q.double().numpy(), k.double().numpy(), kv_seq, window)
    return q, k, go, torch.from_numpy(lse).float()


def run(dg, q, k, go, lse, params, dtype, dv_offset=0):
    dev = torch.device("cuda")
    kv = mha.kv_len(params.q_seq, params.kv_seq)
    n = kv * params.num_kv_heads * params.head_dim
    buf = torch.full((n + dv_offset,), float("nan"), device=dev)
    dv = buf[dv_offset:].view(kv, params.num_kv_heads, params.head_dim)
    dg.mha_grad_v(q.to(dev), k.to(dev), go.to(dev), lse.to(dev), dv, params, dg.DTYPE_CODE[dtype])
    rc = dg.mha_grad_v_check_errors()
    assert rc == 0, dg.STATUS.get(rc, rc)
    return dv.cpu().double().numpy()


def check(got, q, k, go, lse, params, c):
    qd, kd, god, ld = q.double().numpy(), k.double().numpy(), go.double().numpy(), lse.double().numpy()
    ref = mha.grad_v(qd, kd, god, ld, params.kv_seq, params.window_size)
    mag = mha.grad_v(qd, kd, np.abs(god), ld, params.kv_seq, params.window_size)
    bound = c * mag + 1e-6 * np.abs(ref).max()
    assert np.isfinite(got).all()
    worst = float(np.max(np.abs(got - ref) - bound))
    assert worst <= 0, f"error above the bound by {worst:.3g}"
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


# (q_seq, kv_seq, num_heads, num_kv_heads, head_dim, window): causal, full,
# grouped, windowed, ragged lengths, head_dim off 64.
CASES = [
    (64, 0, 4, 2, 64, 0), (100, 0, 8, 2, 64, 0), (77, 90, 4, 4, 64, 0), (130, 0, 6, 3, 64, 17),
    (50, 70, 2, 1, 32, 9), (33, 0, 4, 1, 80, 0), (1, 1, 1, 1, 64, 0), (200, 0, 8, 8, 128, 0),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("case", CASES)
def test_cuda_core_kernel(dg, dtype, case, parity_log):
    q, k, go, lse = make_inputs(*case, dtype, seed=sum(case))
    p = dg.MhaParams(*case)
    dg.mha_grad_v_set_kernel(dg.DGRAD_KERNEL_SIMT)
    try:
        got = run(dg, q, k, go, lse, p, dtype)
    finally:
        dg.mha_grad_v_set_kernel(dg.DGRAD_KERNEL_AUTO)
    err = check(got, q, k, go, lse, p, 1e-4)
    parity_log(f"mha_grad_v simt {dtype} {case}", err, 1e-4)


def test_dv_off_alignment_and_guard(dg):
    case = (40, 0, 2, 1, 64, 0)
    q, k, go, lse = make_inputs(*case, "f32", seed=2)
    p = dg.MhaParams(*case)
    got = run(dg, q, k, go, lse, p, "f32", dv_offset=1)
    check(got, q, k, go, lse, p, 1e-4)


# Tensor-core cases (head_dim 64, an even number of heads): one unit; several
# query blocks under a causal mask (diagonal block masked); full attention with
# ragged lengths; a window; grouped heads; a single position.
TC_CASES = [
    (64, 0, 4, 2, 64, 0), (300, 0, 8, 2, 64, 0), (200, 330, 4, 4, 64, 0), (257, 0, 6, 3, 64, 100),
    (1, 1, 2, 1, 64, 0), (129, 0, 2, 1, 64, 1), (500, 260, 8, 4, 64, 50),
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("case", TC_CASES)
def test_tensor_core_kernel(dg, dtype, case, parity_log):
    q, k, go, lse = make_inputs(*case, dtype, seed=3 * sum(case))
    p = dg.MhaParams(*case)
    dev = torch.device("cuda")
    kv = mha.kv_len(case[0], case[1])
    assert dg.mha_grad_v_select_kernel(q.to(dev), k.to(dev), go.to(dev), lse.to(dev),
                                       torch.empty(kv, case[3], 64, device=dev), p,
                                       dg.DTYPE_CODE[dtype]) == dg.DGRAD_KERNEL_TC
    got = run(dg, q, k, go, lse, p, dtype)
    err = check(got, q, k, go, lse, p, C_TC[dtype])
    parity_log(f"mha_grad_v tc {dtype} {case}", err, C_TC[dtype])


def test_tensor_core_kernel_more_units_than_sms(dg, parity_log):
    """160 units (20 key tiles x 8 KV heads) for 152 SMs: the last key tile runs
    as some CTAs' second unit (K buffer reuse, dV buffer handover, barrier
    phases carried across units).  The oracle checks three key tiles, the last
    among them."""
    case = (2560, 0, 16, 8, 64, 0)
    q, k, go, lse = make_inputs(*case, "bf16", seed=21)
    p = dg.MhaParams(*case)
    got = run(dg, q, k, go, lse, p, "bf16")
    qd, kd, god, ld = q.double().numpy(), k.double().numpy(), go.double().numpy(), lse.double().numpy()
    worst = 0.0
    for t0 in (0, 1280, 2432):
        ref = mha.grad_v_rows(qd, kd, god, ld, 0, 0, t0, t0 + 128)
        mag = mha.grad_v_rows(qd, kd, np.abs(god), ld, 0, 0, t0, t0 + 128)
        bound = C_TC["bf16"] * mag + 1e-6 * np.abs(ref).max()
        err = np.abs(got[t0:t0 + 128] - ref)
        assert (err <= bound).all(), f"key tile {t0}: error above the bound"
        worst = max(worst, float(err.max() / np.abs(ref).max()))
    parity_log("mha_grad_v tc bf16 (2560, 0, 16, 8, 64, 0), 3 key tiles", worst, C_TC["bf16"])


def test_odd_head_count_runs_on_cuda_cores(dg, parity_log):
    """An odd number of query heads (here 3 over one KV head) leaves the
    tensor-core kernel's statistics view without 16-byte rows: auto selection
    takes the CUDA-core kernel, which must still meet its bound."""
    case = (150, 0, 3, 1, 64, 0)
    q, k, go, lse = make_inputs(*case, "bf16", seed=5)
    p = dg.MhaParams(*case)
    dev = torch.device("cuda")
    assert dg.mha_grad_v_select_kernel(q.to(dev), k.to(dev), go.to(dev), lse.to(dev),
                                       torch.empty(150, 1, 64, device=dev), p,
                                       dg.DTYPE_CODE["bf16"]) == dg.DGRAD_KERNEL_SIMT
    got = run(dg, q, k, go, lse, p, "bf16")
    err = check(got, q, k, go, lse, p, 1e-4)
    parity_log("mha_grad_v auto, odd heads bf16 (150, 0, 3, 1, 64, 0)", err, 1e-4)
