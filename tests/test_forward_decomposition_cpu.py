"""The strided forward convolution as one stride-1 valid correlation, checked
on the CPU against the oracle.

conv2d_forward at stride s > 1 runs on the stride-1 path: with u = kh - ph =
s*j + r (floor division), input row s*oh - ph + kh = s*(oh + j) + r, so

    out[n,co,oh,ow] = sum over (r, c, ci, j', i') of
        X''[n, (r,c,ci), oh + j', ow + i'] * W''[co, (r,c,ci), j', i']

with X''[n,(r,c,ci),a,b] = x[n, ci, s*(a + j_min) + r, s*(b + i_min) + c]
(zero outside the image), W''[co,(r,c,ci),j',i'] = w[co, ci, s*(j' + j_min)
+ r + ph, s*(i' + i_min) + c + pw] (zero outside the kernel), j_min =
floor(-ph / s), KH' = floor((kH-1-ph)/s) - j_min + 1, and only the residues r
(c) that some tap reaches.  X'' has OH + KH' - 1 rows, so the correlation
needs no padding.  This restates that identity in numpy and compares it with
the oracle's direct strided forward convolution (a loop over outputs), so a
wrong offset, residue or kernel index in the reading fails here, on the CPU.
"""
import numpy as np
import pytest

import oracle


def residues(k, p, s):
    return sorted({(t - p) % s for t in range(k)})


def decompose(x, w, s, ph, pw):
    """(X'', W'', OH, OW) of the identity above, in float64."""
    N, Ci, H, W = x.shape
    Co, _, kH, kW = w.shape
    OH, OW = (H + 2 * ph - kH) // s + 1, (W + 2 * pw - kW) // s + 1
    rr, cc = residues(kH, ph, s), residues(kW, pw, s)
    jmin, imin = (-ph) // s, (-pw) // s
    KH, KW = (kH - 1 - ph) // s - jmin + 1, (kW - 1 - pw) // s - imin + 1
    Hx, Wx = OH + KH - 1, OW + KW - 1
    X = np.zeros((N, len(rr) * len(cc) * Ci, Hx, Wx))
    Wt = np.zeros((Co, len(rr) * len(cc) * Ci, KH, KW))
    for pr, r in enumerate(rr):
        for pc, c in enumerate(cc):
            base = (pr * len(cc) + pc) * Ci
            for a in range(Hx):
                ih = s * (a + jmin) + r
                if not 0 <= ih < H:
                    continue
                for b in range(Wx):
                    iw = s * (b + imin) + c
                    if 0 <= iw < W:
                        X[:, base:base + Ci, a, b] = x[:, :, ih, iw]
            for j in range(KH):
                kh = s * (j + jmin) + r + ph
                if not 0 <= kh < kH:
                    continue
                for i in range(KW):
                    kw = s * (i + imin) + c + pw
                    if 0 <= kw < kW:
                        Wt[:, base:base + Ci, j, i] = w[:, :, kh, kw]
    return X, Wt, OH, OW


CASES = [
    # (N, Ci, H, W, Co, kH, kW, s, ph, pw)
    (2, 3, 9, 10, 4, 3, 3, 2, 1, 1),
    (1, 2, 8, 8, 3, 1, 1, 2, 0, 0),
    (2, 3, 15, 13, 2, 7, 7, 2, 3, 3),
    (1, 4, 11, 9, 3, 3, 2, 3, 2, 0),
    (1, 2, 17, 13, 2, 2, 2, 4, 1, 0),
    (2, 2, 7, 8, 3, 5, 3, 2, 0, 2),
    (1, 3, 6, 6, 2, 1, 1, 3, 1, 1),   # padding at the kernel size, stride above it
    (1, 2, 9, 9, 2, 4, 4, 2, 3, 3),   # padding k - 1
]


@pytest.mark.parametrize("case", CASES)
def test_strided_forward_is_one_stride1_valid_correlation(case):
    N, Ci, H, W, Co, kH, kW, s, ph, pw = case
    rng = np.random.default_rng(sum(case))
    x = rng.uniform(-1, 1, (N, Ci, H, W))
    w = rng.uniform(-1, 1, (Co, Ci, kH, kW))
    X, Wt, OH, OW = decompose(x, w, s, ph, pw)
    got = oracle.conv2d_forward(X, Wt, 1, 0, 0)
    ref = oracle.conv2d_forward(x, w, s, ph, pw)
    assert got.shape == ref.shape == (N, Co, OH, OW)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_one_by_one_stride_two_keeps_one_residue():
    # A 1x1 stride-2 layer reads residue (0, 0) only: X'' is x decimated, no zero taps.
    x = np.arange(2 * 3 * 8 * 8, dtype=np.float64).reshape(2, 3, 8, 8)
    w = np.ones((4, 3, 1, 1))
    X, Wt, OH, OW = decompose(x, w, 2, 0, 0)
    assert X.shape == (2, 3, 4, 4) and Wt.shape == (4, 3, 1, 1)
    assert np.array_equal(X, x[:, :, ::2, ::2])
