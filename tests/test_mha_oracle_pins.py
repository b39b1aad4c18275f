"""Pins of the attention dV oracle to facts other than its own formula.

The oracle (oracle/mha_grad_v_oracle.c) restates the mha_grad_v.wgsl page:
dV[t][g] = sum over query positions pos (causal: pos >= t; window w > 0:
pos < t + w) and the heads h of KV head g's group of P * dO[pos][h], with
P = exp(min(s - max, 0) - log_sum), s = Q[pos][h] . K[t][g] / sqrt(d) and
(max, log_sum) the forward statistics.  These tests check it against
  * a hand-worked example, full and causal (tests/golden/mha_grad_v_hand.json),
  * torch (float64, CPU): softmax of the masked scores, then P^T dO summed
    over each group's heads -- the library's own softmax and matmul,
  * softmax normalisation: with dO = 1 the sum of dV over key positions is
    the number of (query, head) pairs of the group,
  * grouped-query equivalence: a KV head shared by two query heads equals the
    sum of two single-head problems with that K,
  * the exponent clamp: a max below the score caps P at exp(-log_sum),
and plant mistakes in the oracle source, each of which some pin catches.
"""
import json
import os
import re

import numpy as np
import pytest

from oracle import build_library
from oracle import mha

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mha_grad_v_hand.json")


def _check_golden(lib):
    g = json.load(open(GOLDEN))
    ok = True
    for case in ("full", "causal"):
        c = g[case]
        dv = mha.grad_v(g["q"], g["k"], g["d_out"], c["lse"], c["kv_seq"], c["window"], lib=lib)
        ok = ok and np.allclose(dv, np.asarray(c["dv"]), rtol=0, atol=1e-12)
        lse = mha.forward_lse(g["q"], g["k"], c["kv_seq"], c["window"], lib=lib)
        ok = ok and np.allclose(lse, np.asarray(c["lse"]), rtol=0, atol=1e-12)
    return ok


def test_hand_worked_golden():
    g = json.load(open(GOLDEN))
    assert g["cite"] and g["notes"]
    assert _check_golden(None)


def _rand(q_seq, kv_seq, nh, nkv, hd, seed):
    rng = np.random.default_rng(seed)
    kv = mha.kv_len(q_seq, kv_seq)
    q = rng.normal(size=(q_seq, nh, hd))
    k = rng.normal(size=(kv, nkv, hd))
    go = rng.normal(size=(q_seq, nh, hd))
    return q, k, go


def _torch_case(lib, q_seq, kv_seq, nh, nkv, hd, window, seed):
    torch = pytest.importorskip("torch")
    q, k, go = _rand(q_seq, kv_seq, nh, nkv, hd, seed)
    kv = mha.kv_len(q_seq, kv_seq)
    lse = mha.forward_lse(q, k, kv_seq, window, lib=lib)
    dv = mha.grad_v(q, k, go, lse, kv_seq, window, lib=lib)
    hpk = nh // nkv
    pos = torch.arange(q_seq)[:, None]
    t = torch.arange(kv)[None, :]
    allowed = torch.ones(q_seq, kv, dtype=torch.bool)
    if kv_seq == 0:
        allowed &= t <= pos
    if window > 0:
        allowed &= t > pos - window
    want = torch.zeros(kv, nkv, hd, dtype=torch.float64)
    for h in range(nh):
        g = h // hpk
        s = torch.from_numpy(q[:, h, :]) @ torch.from_numpy(k[:, g, :]).T / np.sqrt(hd)
        s = s.masked_fill(~allowed, float("-inf"))
        p = torch.softmax(s, dim=1)
        p = torch.nan_to_num(p, nan=0.0)  # a query that attends no key contributes nothing
        want[:, g, :] += p.T @ torch.from_numpy(go[:, h, :])
    return np.allclose(dv, want.numpy(), rtol=1e-11, atol=1e-11)


TORCH_CASES = [
    (5, 7, 2, 2, 4, 0), (6, 0, 4, 2, 8, 0), (9, 0, 6, 2, 3, 3), (8, 11, 4, 1, 5, 4), (1, 1, 1, 1, 1, 0),
    (16, 0, 8, 8, 16, 1), (12, 12, 4, 4, 64, 0),
]


@pytest.mark.parametrize("case", TORCH_CASES)
def test_matches_torch_softmax_then_matmul(case):
    assert _torch_case(None, *case, seed=sum(case))


def _normalisation_case(lib, q_seq, kv_seq, nh, nkv, hd, window, seed):
    q, k, _ = _rand(q_seq, kv_seq, nh, nkv, hd, seed)
    lse = mha.forward_lse(q, k, kv_seq, window, lib=lib)
    dv = mha.grad_v(q, k, np.ones((q_seq, nh, hd)), lse, kv_seq, window, lib=lib)
    # every query attends at least one key here (causal: itself; full: all)
    return np.allclose(dv.sum(axis=0), q_seq * (nh // nkv), rtol=1e-12)


def test_softmax_normalisation():
    for case in ((7, 0, 4, 2, 5, 0), (7, 9, 2, 1, 3, 0), (10, 0, 4, 4, 6, 3)):
        assert _normalisation_case(None, *case, seed=3)


def _gqa_case(lib, seed=0):
    q, k, go = _rand(6, 0, 2, 1, 4, seed)
    lse = mha.forward_lse(q, k, 0, 0, lib=lib)
    dv = mha.grad_v(q, k, go, lse, 0, 0, lib=lib)
    parts = sum(mha.grad_v(q[:, h:h + 1], k, go[:, h:h + 1], lse[:, h:h + 1], 0, 0, lib=lib) for h in range(2))
    return np.allclose(dv, parts, rtol=1e-12, atol=1e-12)


def test_grouped_query_equals_sum_of_single_heads():
    assert _gqa_case(None)


def _clamp_case(lib):
    # one query, one key, head_dim 1: s = 2 * 3 = 6 > max = 1; log_sum = ln 2 -> P = exp(0 - ln 2) = 1/2
    dv = mha.grad_v([[[2.0]]], [[[3.0]]], [[[5.0]]], [[[1.0, np.log(2.0)]]], 1, 0, lib=lib)
    return np.allclose(dv, [[[2.5]]], rtol=0, atol=1e-12)


def test_exponent_clamp():
    assert _clamp_case(None)


def _pins_pass(lib):
    try:
        return (_check_golden(lib) and _torch_case(lib, 9, 0, 6, 2, 3, 3, 1) and _torch_case(lib, 8, 11, 4, 1, 5, 4, 2)
                and _torch_case(lib, 5, 7, 4, 2, 4, 0, 5) and _normalisation_case(lib, 7, 0, 4, 2, 5, 0, 3)
                and _gqa_case(lib) and _clamp_case(lib))
    except (ValueError, AssertionError, FloatingPointError):
        return False


def test_unmutated_oracle_passes_the_pins():
    assert _pins_pass(None)


# Planted mistakes: each mutant of the oracle source must fail some pin.
MUTANTS = {
    "no_scale": ("s *= scale;\n                    const double *st", "const double *st"),
    "causal_start_after_t": ("const int start = causal ? t : 0;", "const int start = causal ? t + 1 : 0;"),
    "window_one_longer": ("if (window > 0 && t + window < end) end = t + window;",
                          "if (window > 0 && t + window + 1 < end) end = t + window + 1;"),
    "heads_interleaved": ("const int h = g * hpk + r;", "const int h = r * num_kv_heads + g;"),
    "clamp_dropped": ("if (e > 0.0) e = 0.0;", ""),
    "lse_halves_swapped": ("double e = s - st[0];", "double e = s - st[1];"),
    "d_out_of_kv_head": ("const double *go = d_out + pos * q_dim + (int64_t)h * head_dim;",
                         "const double *go = d_out + pos * q_dim + (int64_t)g * head_dim;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mutant_is_caught(name, tmp_path):
    src = open(mha.SOURCE).read()
    old, new = MUTANTS[name]
    assert old in src, f"mutant site of {name} not found"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new, 1))
    lib = mha.load_library(build_library(str(mutated), str(tmp_path / "libmutant.so")))
    assert not _pins_pass(lib), f"mutant {name} slipped through every pin"


def test_mutant_sites_are_distinct():
    assert len({m[0] + "->" + m[1] for m in MUTANTS.values()}) == len(MUTANTS)


def test_row_range_matches_the_full_result():
    q, k, go = _rand(20, 0, 4, 2, 8, 11)
    lse = mha.forward_lse(q, k, 0, 5)
    full = mha.grad_v(q, k, go, lse, 0, 5)
    for a, b in ((0, 20), (3, 9), (19, 20), (7, 7)):
        assert np.array_equal(mha.grad_v_rows(q, k, go, lse, 0, 5, a, b), full[a:b])
