"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin below is independent of the oracle's own code:
  * hand-worked fixtures (tests/golden/*.json, each with its derivation),
  * closed-form tap counts for all-ones inputs, enumerated from the forward
    side (over output rows) rather than the gather side (over taps),
  * torch's CPU float64 conv2d and conv2d_input (a third-party routine),
  * numpy matmul for the 1x1 stride-1 unpadded case (a pure GEMM),
  * the adjoint identity <conv(x), g> = <x, dgrad(g)> against the separately
    written forward oracle, and finite differences of that forward,
  * planted mutants of the oracle source, each of which some pin must catch.
"""
import glob
import json
import os
import re

import numpy as np
import pytest
import torch

import oracle
from conv2d_backward_implicit_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return workloads.make_tensor(shape, seed, "f32", "uniform").double().numpy()


def _case(shape_tuple, seed):
    N, Ci, H, W, Co, kH, kW, s, ph, pw = shape_tuple
    OH = oracle.out_size(H, kH, ph, s)
    OW = oracle.out_size(W, kW, pw, s)
    g = _rand((N, Co, OH, OW), seed)
    w = _rand((Co, Ci, kH, kW), seed + 1)
    return g, w, (N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW)


SWEEP = workloads.random_small_shapes(160, seed=7)


# --------------------------------------------------------------------------
@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(GOLDEN, "hand_*.json"))),
                         ids=lambda p: os.path.basename(p))
def test_golden_fixture(path):
    fx = json.load(open(path))
    p = fx["params"]
    g = np.array(fx["grad_out"], dtype=np.float64)
    w = np.array(fx["weight"], dtype=np.float64)
    assert g.shape == (p["N"], p["Co"], p["OH"], p["OW"])
    assert w.shape == (p["Co"], p["Ci"], p["kH"], p["kW"])
    assert oracle.out_size(p["H"], p["kH"], p["padding_h"], p["stride"]) == p["OH"]
    assert oracle.out_size(p["W"], p["kW"], p["padding_w"], p["stride"]) == p["OW"]
    got = oracle.dgrad(g, w, p["H"], p["W"], p["stride"], p["padding_h"], p["padding_w"])
    np.testing.assert_array_equal(got, np.array(fx["grad_in"], dtype=np.float64))


def test_out_size_closed_form():
    # (H + 2p - k) // s + 1 on the five workloads' sizes, and the no-fit case.
    for wl in workloads.ALL:
        assert oracle.out_size(wl.H, wl.kH, wl.padding_h, wl.stride) == wl.OH
        assert oracle.out_size(wl.W, wl.kW, wl.padding_w, wl.stride) == wl.OW
    assert oracle.out_size(2, 5, 1, 1) == 0
    assert oracle.out_size(7, 2, 0, 3) == 2  # floor: rows 0..3, 3..5 fit; 6 is left over


def _covering_count(size, k, pad, s, out):
    """How many (output row, tap) pairs touch each input row, counted over output rows."""
    cnt = np.zeros(size, dtype=np.int64)
    for o in range(out):
        for kk in range(k):
            y = o * s - pad + kk
            if 0 <= y < size:
                cnt[y] += 1
    return cnt


@pytest.mark.parametrize("shape", SWEEP[:60])
def test_all_ones_closed_form(shape):
    N, Ci, H, W, Co, kH, kW, s, ph, pw = shape
    OH, OW = oracle.out_size(H, kH, ph, s), oracle.out_size(W, kW, pw, s)
    g = np.ones((N, Co, OH, OW))
    w = np.ones((Co, Ci, kH, kW))
    got = oracle.dgrad(g, w, H, W, s, ph, pw)
    ch = _covering_count(H, kH, ph, s, OH)
    cw = _covering_count(W, kW, pw, s, OW)
    want = Co * np.outer(ch, cw)
    np.testing.assert_array_equal(got, np.broadcast_to(want, got.shape))


def test_all_ones_interior_is_full_kernel():
    # Stride 1, interior pixel: every one of the kH*kW taps lands, times Co.
    g = np.ones((1, 3, 9, 9))
    w = np.ones((3, 2, 3, 5))
    got = oracle.dgrad(g, w, 9, 11, 1, 1, 2)  # OH=9, OW=11
    assert got[0, 1, 4, 5] == 3 * 3 * 5


@pytest.mark.parametrize("idx", range(0, 160, 1))
def test_against_torch_conv2d_input(idx):
    g, w, (N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW) = _case(SWEEP[idx], 100 + idx)
    got = oracle.dgrad(g, w, H, W, s, ph, pw)
    want = torch.nn.grad.conv2d_input((N, Ci, H, W), torch.from_numpy(w), torch.from_numpy(g),
                                      stride=s, padding=(ph, pw)).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("idx", range(0, 160, 4))
def test_forward_against_torch_conv2d(idx):
    N, Ci, H, W, Co, kH, kW, s, ph, pw = SWEEP[idx]
    x = _rand((N, Ci, H, W), 500 + idx)
    w = _rand((Co, Ci, kH, kW), 900 + idx)
    got = oracle.conv2d_forward(x, w, s, ph, pw)
    want = torch.nn.functional.conv2d(torch.from_numpy(x), torch.from_numpy(w), stride=s,
                                      padding=(ph, pw)).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_pointwise_is_matmul():
    # 1x1, stride 1, no padding: grad_in[n] = W^T @ G[n] with G[n] = [Co, H*W].
    N, Ci, Co, H, W = 3, 7, 5, 4, 6
    g = _rand((N, Co, H, W), 11)
    w = _rand((Co, Ci, 1, 1), 12)
    got = oracle.dgrad(g, w, H, W, 1, 0, 0)
    Wm = w[:, :, 0, 0]
    want = np.stack([(Wm.T @ g[n].reshape(Co, H * W)).reshape(Ci, H, W) for n in range(N)])
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("idx", range(160))
def test_adjoint_identity_sweep(idx):
    g, w, (N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW) = _case(SWEEP[idx], 3000 + idx)
    x = _rand((N, Ci, H, W), 7000 + idx)
    lhs = float(np.sum(oracle.conv2d_forward(x, w, s, ph, pw) * g))
    rhs = float(np.sum(x * oracle.dgrad(g, w, H, W, s, ph, pw)))
    scale = float(np.sum(np.abs(x)) * np.max(np.abs(w)) * max(1.0, np.max(np.abs(g)))) + 1e-300
    assert abs(lhs - rhs) <= 1e-10 * max(abs(lhs), 1e-3 * scale)


@pytest.mark.parametrize("wl", workloads.ALL, ids=lambda w: w.name)
def test_adjoint_identity_workloads(wl):
    # The five workloads' per-image shapes, with one batch item (two for the tiny one).
    small = wl.with_batch(1 if wl.N > 1 else wl.N)
    g, w = workloads.make_inputs(small, seed=0)
    g, w = g.double().numpy(), w.double().numpy()
    x = workloads.make_tensor(small.grad_in_shape, 99, "f32", "normal").double().numpy()
    # Keep the forward pass cheap: restrict to a few input channels for the big ones.
    ci_keep = min(small.Ci, 8)
    w = w[:, :ci_keep]
    x = x[:, :ci_keep]
    lhs = float(np.sum(oracle.conv2d_forward(x, w, wl.stride, wl.padding_h, wl.padding_w) * g))
    rhs = float(np.sum(x * oracle.dgrad(g, w, wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)))
    assert abs(lhs - rhs) <= 1e-10 * abs(lhs)


def test_finite_differences():
    # L(x) = <conv(x), g> is linear in x, so the central difference with step 1
    # at coordinate i equals dgrad(g)[i] up to double rounding.
    N, Ci, H, W, Co, kH, kW, s, ph, pw = 2, 3, 7, 6, 4, 3, 2, 2, 1, 0
    OH, OW = oracle.out_size(H, kH, ph, s), oracle.out_size(W, kW, pw, s)
    g = _rand((N, Co, OH, OW), 21)
    w = _rand((Co, Ci, kH, kW), 22)
    x = _rand((N, Ci, H, W), 23)
    dg = oracle.dgrad(g, w, H, W, s, ph, pw)
    rng = np.random.default_rng(5)
    for _ in range(40):
        i = tuple(int(rng.integers(0, d)) for d in x.shape)
        xp, xm = x.copy(), x.copy()
        xp[i] += 1.0
        xm[i] -= 1.0
        fd = (np.sum(oracle.conv2d_forward(xp, w, s, ph, pw) * g)
              - np.sum(oracle.conv2d_forward(xm, w, s, ph, pw) * g)) / 2.0
        assert abs(fd - dg[i]) <= 1e-9 * max(1.0, abs(dg[i]))


def test_points_match_full():
    g, w, (N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW) = _case((2, 3, 9, 8, 4, 5, 3, 2, 2, 1), 41)
    full = oracle.dgrad(g, w, H, W, s, ph, pw)
    rng = np.random.default_rng(0)
    pts = np.stack([rng.integers(0, d, 50) for d in full.shape], axis=1)
    got = oracle.dgrad_points(g, w, pts, H, W, s, ph, pw)
    np.testing.assert_array_equal(got, full[tuple(pts.T)])


def test_thread_count_does_not_change_bits():
    g, w, (N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW) = _case((2, 6, 9, 9, 5, 3, 3, 1, 1, 1), 43)
    a = oracle.dgrad(g, w, H, W, s, ph, pw, nthreads=1)
    b = oracle.dgrad(g, w, H, W, s, ph, pw, nthreads=7)
    np.testing.assert_array_equal(a, b)


# --------------------------------------------------------------------------
# The page's stride-1 index shortcut agrees with the definition only when
# kernel-1 == 2*padding on both axes; for stride > 1 it is the definition.
@pytest.mark.parametrize("idx", range(0, 160, 2))
def test_shader_index_map_agreement(idx):
    g, w, (N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW) = _case(SWEEP[idx], 5000 + idx)
    ref = oracle.dgrad(g, w, H, W, s, ph, pw)
    sh = oracle.shader_index_dgrad(g, w, H, W, s, ph, pw)
    if s > 1 or (kH - 1 == 2 * ph and kW - 1 == 2 * pw):
        np.testing.assert_allclose(sh, ref, rtol=1e-13, atol=1e-13)


def test_shader_index_map_diverges_off_centre():
    path = os.path.join(GOLDEN, "hand_2x2_s1_p0.json")
    fx = json.load(open(path))
    p = fx["params"]
    g = np.array(fx["grad_out"], dtype=np.float64)
    w = np.array(fx["weight"], dtype=np.float64)
    sh = oracle.shader_index_dgrad(g, w, p["H"], p["W"], 1, 0, 0)
    assert not np.array_equal(sh, np.array(fx["grad_in"], dtype=np.float64))
    # 3x3 with padding 0 (kH-1 = 2 != 0): also different from the definition.
    g2, w2, dims = _case((1, 2, 6, 6, 2, 3, 3, 1, 0, 0), 77)
    ref = oracle.dgrad(g2, w2, 6, 6, 1, 0, 0)
    assert not np.allclose(oracle.shader_index_dgrad(g2, w2, 6, 6, 1, 0, 0), ref)


# --------------------------------------------------------------------------
# Planted mistakes: each mutant of the oracle source must fail some pin.
MUTANTS = {
    "sign_of_padding": ("int th = ih + p->ph - kh;", "int th = ih - p->ph + kh;"),
    "flipped_tap": ("w[idx4(co, ci, kh, kw, p->Ci, p->kH, p->kW)]",
                    "w[idx4(co, ci, p->kH - 1 - kh, kw, p->Ci, p->kH, p->kW)]"),
    "dropped_divisibility": ("if (tw < 0 || tw % p->s != 0) continue;", "if (tw < 0) continue;"),
    "dropped_channel": ("for (int co = 0; co < p->Co; ++co) {", "for (int co = 1; co < p->Co; ++co) {"),
    "padding_axis_swap": ("int tw = iw + p->pw - kw;", "int tw = iw + p->ph - kw;"),
    "transposed_channels": ("w[idx4(co, ci, kh, kw, p->Ci, p->kH, p->kW)]",
                            "w[idx4(ci % p->Co, co % p->Ci, kh, kw, p->Ci, p->kH, p->kW)]"),
}


def _pins_pass(lib) -> bool:
    """Run a compact set of the pins above against another build of the oracle."""
    for path in sorted(glob.glob(os.path.join(GOLDEN, "hand_*.json"))):
        fx = json.load(open(path))
        p = fx["params"]
        got = oracle.dgrad(np.array(fx["grad_out"], float), np.array(fx["weight"], float),
                           p["H"], p["W"], p["stride"], p["padding_h"], p["padding_w"], lib=lib)
        if not np.array_equal(got, np.array(fx["grad_in"], float)):
            return False
    for idx in range(0, 160, 5):
        g, w, (N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW) = _case(SWEEP[idx], 100 + idx)
        got = oracle.dgrad(g, w, H, W, s, ph, pw, lib=lib)
        want = torch.nn.grad.conv2d_input((N, Ci, H, W), torch.from_numpy(w), torch.from_numpy(g),
                                          stride=s, padding=(ph, pw)).numpy()
        if not np.allclose(got, want, rtol=1e-12, atol=1e-12):
            return False
    return True


def test_unmutated_source_passes_compact_pins():
    assert _pins_pass(oracle.load_library())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mutant_is_caught(name, tmp_path):
    src = open(oracle.SOURCE).read()
    old, new = MUTANTS[name]
    # Mutate only inside dgrad_one, the definition's inner loop.
    start = src.index("static double dgrad_one(")
    end = src.index("typedef struct {", start)
    body = src[start:end]
    assert body.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = src[:start] + body.replace(old, new) + src[end:]
    c_path = tmp_path / f"mut_{name}.c"
    c_path.write_text(mutated)
    so = oracle.build_library(str(c_path), str(tmp_path / f"libmut_{name}.so"))
    lib = oracle.load_library(so)
    assert not _pins_pass(lib), f"mutant {name} slipped through every pin"


def test_mutant_sites_are_distinct():
    assert len({m[0] + "->" + m[1] for m in MUTANTS.values()}) == len(MUTANTS)
    assert all(re.search(r"\S", m[1]) for m in MUTANTS.values())
