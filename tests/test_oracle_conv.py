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


def _tw_hand_inputs():
    """One 128-channel tile (C_out = 2), C_in = 64, so a group is one whole tap. Tap
    (2, 2) holds 2 at channel 1 of output 1 (group score 2), the centre tap 1 at
    channel 0 of output 0 and -0.5 at channel 3 of output 1 (score 1.5), tap (0, 0)
    0.75 at channel 5 of output 0 (score 0.75); the other taps are zero."""
    Cin, Cout = 64, 2
    Wf = np.zeros((Cout, 9 * Cin))
    Wf[0, 4 * Cin + 0] = 1.0
    Wf[1, 4 * Cin + 3] = -0.5
    Wf[1, 8 * Cin + 1] = 2.0
    Wf[0, 0 * Cin + 5] = 0.75
    rng = np.random.default_rng(9)
    X = rng.integers(-4, 5, size=(1, 2, 3, Cin)) / 4.0
    return _bits(Wf), _bits(X), codecs.decode(_bits(X), "bf16")


def test_tile_wise_filter_hand_case():
    """Kept groups follow the group scores (2 > 1.5 > 0.75 > 0); the result is the
    convolution sum of the kept taps alone, written out here per pixel."""
    Wf, X, x = _tw_hand_inputs()
    H, W = 2, 3
    at = lambda h, w, c: x[0, h, w, c] if 0 <= h < H and 0 <= w < W else 0.0
    for keep, want_groups in ((1, [8]), (2, [4, 8]), (3, [0, 4, 8])):
        Y, _, form = conv.conv3x3_tw(Wf, X, "bf16", "bf16", [keep])
        assert list(form["indices"]) == want_groups
        want = np.zeros((2, H * W))
        for h in range(H):
            for w in range(W):
                if 4 in want_groups:
                    want[0, h * W + w] += at(h, w, 0)
                    want[1, h * W + w] += -0.5 * at(h, w, 3)
                if 8 in want_groups:                      # tap (2, 2): X[h + 1, w + 1]
                    want[1, h * W + w] += 2.0 * at(h + 1, w + 1, 1)
                if 0 in want_groups:                      # tap (0, 0): X[h - 1, w - 1]
                    want[0, h * W + w] += 0.75 * at(h - 1, w - 1, 5)
        assert np.array_equal(codecs.decode(Y, "bf16"), want)


def test_tile_wise_filter_all_and_none_kept():
    rng = np.random.default_rng(11)
    Nb, H, W, Cin, Cout = 1, 3, 4, 64, 200              # two tiles, the second ragged
    X = _bits(rng.integers(-4, 5, size=(Nb, H, W, Cin)) / 4.0)
    Wf = _bits(rng.integers(-4, 5, size=(Cout, 9 * Cin)) / 8.0)
    Y_all, _, _ = conv.conv3x3_tw(Wf, X, "bf16", "bf16", [9, 9])
    Y_dense, _ = conv.conv3x3(Wf, X, "bf16", "bf16", sparse=False)
    assert np.array_equal(Y_all, Y_dense)
    Y_none, B_none, _ = conv.conv3x3_tw(Wf, X, "bf16", "bf16", [0, 0])
    assert not codecs.decode(Y_none, "bf16").any() and not B_none.any()


def test_tile_wise_filter_keeps_the_top_groups_per_tile():
    """Brute force on the group scores in fp64: each tile keeps the keep[t] groups of
    largest sum |w| (ties to the lower group), and the masked filter is zero
    exactly outside them."""
    rng = np.random.default_rng(12)
    Cin, Cout = 128, 256
    Wf = _bits(rng.standard_normal((Cout, 9 * Cin)))
    keep = [5, 11]
    X = _bits(rng.standard_normal((1, 2, 2, Cin)))
    _, _, form = conv.conv3x3_tw(Wf, X, "bf16", "bf16", keep)
    w = np.abs(codecs.decode(Wf, "bf16"))
    for t in range(2):
        score = w[128 * t:128 * (t + 1)].reshape(128, 18, 64).sum(axis=(0, 2))
        order = sorted(range(18), key=lambda g: (-score[g], g))
        got = form["indices"][form["offsets"][t]:form["offsets"][t + 1]]
        assert sorted(order[:keep[t]]) == list(got)
