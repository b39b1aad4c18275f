"""Pins of the RMSNorm + matmul oracle to facts other than its own formula.

The oracle (oracle/rmsnorm_matmul_oracle.c) restates the definition on the
matmul_rms_norm.wgsl page: C = RmsNorm(X, W_norm) x W_proj with
RmsNorm(X, W_norm)[i, t] = X[i, t] * W_norm[t] / sqrt(mean_t X[i, t]^2 + eps).
These tests check it against
  * two hand-worked examples (tests/golden/rmsnorm_*.json, derivations inside),
  * a special case that reduces to a library matmul: rows of +-1 have mean
    square 1, so with eps = 0 the norm is the identity and C = (X W_norm) W_proj,
  * a closed form with eps: constant rows c give r = 1 / sqrt(c^2 + eps),
  * invariants: with eps = 0, C(a X) = C(X) for a > 0 and C(-X) = -C(X),
  * torch's own rms_norm (float64, CPU) followed by a matmul,
and plant six mistakes in the oracle source, each of which some pin catches.
"""
import json
import os
import re

import numpy as np
import pytest

from oracle import build_library
from oracle import rmsnorm as orn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _check_golden(lib, name):
    g = _golden(name)
    c = orn.rmsnorm_matmul(g["x"], g["w_norm"], g["w_proj"], g["eps"], lib=lib)
    return c.shape == (g["m"], g["n"]) and np.allclose(c, np.asarray(g["c"], dtype=np.float64), rtol=0, atol=1e-12)


@pytest.mark.parametrize("name", ["rmsnorm_hand_unit_rms.json", "rmsnorm_hand_eps.json"])
def test_hand_worked_golden(name):
    g = _golden(name)
    assert g["cite"] and g["notes"]
    assert _check_golden(None, name)


def _unit_rms_case(lib, seed=0, m=7, k=12, n=5):
    rng = np.random.default_rng(seed)
    x = rng.choice([-1.0, 1.0], size=(m, k))
    wn = rng.uniform(-2, 2, k)
    wp = rng.uniform(-1, 1, (k, n))
    c = orn.rmsnorm_matmul(x, wn, wp, 0.0, lib=lib)
    return np.allclose(c, (x * wn[None, :]) @ wp, rtol=1e-12, atol=1e-12)


def test_unit_rms_rows_reduce_to_a_matmul():
    for seed in range(4):
        assert _unit_rms_case(None, seed)


def _eps_closed_form_case(lib, seed=0, m=5, k=9, n=4):
    rng = np.random.default_rng(seed + 100)
    cst = rng.uniform(0.5, 3.0, m) * rng.choice([-1.0, 1.0], m)
    x = np.repeat(cst[:, None], k, axis=1)
    eps = 0.75
    wn = rng.uniform(-2, 2, k)
    wp = rng.uniform(-1, 1, (k, n))
    r = 1.0 / np.sqrt(cst * cst + eps)
    want = (cst * r)[:, None] * (wn @ wp)[None, :]
    c = orn.rmsnorm_matmul(x, wn, wp, eps, lib=lib)
    rr = orn.rms_rows(x, eps, lib=lib)
    return np.allclose(c, want, rtol=1e-12, atol=1e-12) and np.allclose(rr, r, rtol=1e-14)


def test_constant_rows_closed_form_with_eps():
    for seed in range(3):
        assert _eps_closed_form_case(None, seed)


def _invariants_case(lib, seed=0, m=6, k=20, n=7):
    rng = np.random.default_rng(seed + 200)
    x = rng.normal(size=(m, k))
    wn = rng.normal(size=k)
    wp = rng.normal(size=(k, n))
    c = orn.rmsnorm_matmul(x, wn, wp, 0.0, lib=lib)
    a = rng.uniform(0.01, 100.0)
    ok = np.allclose(orn.rmsnorm_matmul(a * x, wn, wp, 0.0, lib=lib), c, rtol=1e-11, atol=1e-12)
    return ok and np.allclose(orn.rmsnorm_matmul(-x, wn, wp, 0.0, lib=lib), -c, rtol=0, atol=0)


def test_scale_and_sign_invariants():
    for seed in range(3):
        assert _invariants_case(None, seed)


def _torch_case(lib, seed=0, m=9, k=33, n=11, eps=1e-5):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(seed + 300)
    x = rng.normal(size=(m, k)) * rng.uniform(0.1, 10.0, (m, 1))
    wn = rng.normal(size=k)
    wp = rng.normal(size=(k, n))
    xt = torch.from_numpy(x)
    ref = torch.nn.functional.rms_norm(xt, (k,), weight=torch.from_numpy(wn), eps=eps) @ torch.from_numpy(wp)
    c = orn.rmsnorm_matmul(x, wn, wp, eps, lib=lib)
    a = orn.normalize(x, wn, eps, lib=lib)
    return np.allclose(c, ref.numpy(), rtol=1e-12, atol=1e-12) and np.allclose(a @ wp, c, rtol=1e-12, atol=1e-12)


def test_matches_torch_rms_norm_then_matmul():
    for seed in range(4):
        assert _torch_case(None, seed)
    assert _torch_case(None, 9, m=1, k=1, n=1)
    assert _torch_case(None, 10, m=3, k=64, n=130, eps=0.0)


def _pins_pass(lib):
    try:
        return (all(_check_golden(lib, n) for n in ("rmsnorm_hand_unit_rms.json", "rmsnorm_hand_eps.json"))
                and _unit_rms_case(lib) and _eps_closed_form_case(lib) and _invariants_case(lib)
                and _torch_case(lib))
    except (ValueError, AssertionError, FloatingPointError):
        return False


def test_unmutated_oracle_passes_the_pins():
    assert _pins_pass(None)


# Planted mistakes: each mutant of the oracle source must fail some pin.
MUTANTS = {
    "sum_not_mean": ("ss / (double)k + eps", "ss + eps"),
    "eps_outside_root": ("1.0 / sqrt(ss / (double)k + eps)", "1.0 / sqrt(ss / (double)k) + eps"),
    "sqrt_not_rsqrt": ("1.0 / sqrt(", "sqrt("),
    "row_scale_dropped": ("x[(int64_t)i * k + t] * r * w_norm[t]", "x[(int64_t)i * k + t] * w_norm[t]"),
    "w_norm_shifted": ("r * w_norm[t]", "r * w_norm[(i + t) % k]"),
    "w_proj_transposed": ("w_proj[(int64_t)t * n + j]", "w_proj[(int64_t)j * k + t]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mutant_is_caught(name, tmp_path):
    src = open(orn.SOURCE).read()
    old, new = MUTANTS[name]
    assert old in src, f"mutant site of {name} not found"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = orn.load_library(build_library(str(mutated), str(tmp_path / "libmutant.so")))
    assert not _pins_pass(lib), f"mutant {name} slipped through every pin"


def test_mutant_sites_are_distinct():
    assert len({m[0] + "->" + m[1] for m in MUTANTS.values()}) == len(MUTANTS)
    assert all(re.search(r"\S", m[1]) for m in MUTANTS.values())
