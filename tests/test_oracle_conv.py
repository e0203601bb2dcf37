"""Pins for the oracle's 3x3 convolution: the im2col form against the convolution
sum written out with loops, a centre-tap identity, a shifted-tap closed form
(the zero padding at the image border), and a planted tap-order mistake."""
import numpy as np
import pytest

from oracle import codecs, conv, gemm, sp24


def _bits(x, dt="bf16"):
    return codecs.encode(np.asarray(x, dtype=np.float64), dt)


def test_im2col_form_matches_the_direct_sum():
    rng = np.random.default_rng(2)
    Nb, H, W, Cin, Cout = 2, 5, 4, 8, 6
    X = _bits(rng.integers(-4, 5, size=(Nb, H, W, Cin)) / 4.0)
    Wf = _bits(rng.integers(-4, 5, size=(Cout, 9 * Cin)) / 4.0)
    Y, _ = conv.conv3x3(Wf, X, "bf16", "bf16", sparse=False)
    direct = conv.conv3x3_direct(Wf, X, "bf16")
    assert np.array_equal(codecs.decode(Y, "bf16"), direct)        # small dyadic values: exact


def test_centre_tap_is_the_identity():
    rng = np.random.default_rng(3)
    Nb, H, W, Cin = 1, 4, 6, 8
    X = _bits(rng.standard_normal((Nb, H, W, Cin)))
    Wf = np.zeros((Cin, 9 * Cin))
    for c in range(Cin):
        Wf[c, 4 * Cin + c] = 1.0                                    # tap (1, 1): no shift
    Y, _ = conv.conv3x3(_bits(Wf), X, "bf16", "bf16", sparse=False)
    assert np.array_equal(Y, X.reshape(-1, Cin).T)


def test_shifted_tap_and_zero_padding():
    Nb, H, W, Cin = 1, 3, 3, 4
    X = _bits(np.arange(Nb * H * W * Cin).reshape(Nb, H, W, Cin) / 8.0)
    Wf = np.zeros((1, 9 * Cin))
    Wf[0, (3 * 0 + 2) * Cin + 1] = 1.0                              # tap (r, s) = (0, 2), channel 1
    Y, _ = conv.conv3x3(_bits(Wf), X, "bf16", "bf16", sparse=False)
    x = codecs.decode(X, "bf16")[0, :, :, 1]
    want = np.zeros((H, W))
    for h in range(H):
        for w in range(W):                                          # Y[h, w] = X[h - 1, w + 1]
            if h - 1 >= 0 and w + 1 < W:
                want[h, w] = x[h - 1, w + 1]
    assert np.array_equal(codecs.decode(Y, "bf16").reshape(H, W), want)


def test_sparse_filter_is_the_2to4_pruned_filter_and_a_planted_tap_order_fails():
    rng = np.random.default_rng(4)
    Nb, H, W, Cin, Cout = 1, 4, 4, 8, 5
    X = _bits(rng.standard_normal((Nb, H, W, Cin)))
    Wf = _bits(rng.standard_normal((Cout, 9 * Cin)))
    Y, B = conv.conv3x3(Wf, X, "bf16", "bf16", sparse=True)
    Wp = sp24.prune(Wf, "bf16")
    Y2, _ = conv.conv3x3(Wp, X, "bf16", "bf16", sparse=False)
    assert np.array_equal(Y, Y2)
    # tap order (s, r) instead of (r, s): the transposed filter gives another result
    Wt = Wp.reshape(Cout, 3, 3, Cin).transpose(0, 2, 1, 3).reshape(Cout, 9 * Cin)
    Y3, _ = conv.conv3x3(Wt, X, "bf16", "bf16", sparse=False)
    assert not gemm.within_bound(Y3, Y, B, "bf16", 1e-2).all()
