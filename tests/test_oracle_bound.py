"""Pins for the checker itself: the elementwise error bound B = |alpha| sum_k |w x|
that every GPU parity verdict ("|Y - Y_ref| <= rel * B") rests on, and the
reference values Y, for every product form of the oracle. Expected values are
worked out by hand in tests/golden/bound_hand.json (alpha negative, cancellation
in Y, pruned weights that would change B if counted), and planted mistakes in
the bound (a signed alpha, a dropped alpha, the unpruned weights) must fail."""
import json
import os

import numpy as np
import pytest

from oracle import bw, codecs, conv, ew, gemm, sp24, tw

HERE = os.path.dirname(os.path.abspath(__file__))
DT = "bf16"


@pytest.fixture(scope="module")
def fx():
    with open(os.path.join(HERE, "golden", "bound_hand.json")) as f:
        return json.load(f)


def _bits(a):
    return codecs.encode(np.asarray(a, dtype=np.float64), DT)


def _vals(bits):
    return codecs.decode(bits, DT)


def _check_dense(c):
    W, X = _bits(c["W"]), _bits(c["X"])
    assert (_vals(gemm.gemm_dense(W, X, DT, DT, c["alpha"])) == np.array(c["Y"])).all()
    assert (gemm.bound(W, X, DT, c["alpha"]) == np.array(c["B"])).all()


def _check_sp24(c):
    W, X = _bits(c["W"]), _bits(c["X"])
    v, m = sp24.compress(W, DT)
    K = W.shape[1]
    assert (_vals(gemm.gemm_sp24(v, m, K, X, DT, DT, c["alpha"])) == np.array(c["Y"])).all()
    assert (gemm.bound(sp24.decompress(v, m, K), X, DT, c["alpha"]) == np.array(c["B"])).all()


def _tw_W(c):
    W = np.zeros((256, 8))
    for r, row in c["W_rows"].items():
        W[int(r)] = row
    return _bits(W)


def _check_tw(c, tvw):
    W, X = _tw_W(c), _bits(c["X"])
    keep = np.array(c["tvw_keep" if tvw else "tw_keep"], dtype=np.int32)
    form = tw.prune(W, DT, keep, tvw)
    Y, B = tw.gemm(form, keep, X, DT, DT, 256, tvw, c["alpha"])
    rows = c["rows"]
    key = "tvw" if tvw else "tw"
    assert (_vals(Y[rows]) == np.array(c[f"{key}_Y"])).all()
    assert (B[rows] == np.array(c[f"{key}_B"])).all()


def _bw_inputs(c):
    K = c["K"]
    W = np.zeros((256, K))
    for i, k, v in c["entries"]:
        W[i, k] = v
    X = np.full((K, 1), c["X_col"]["default"])
    for k, v in c["X_col"].items():
        if k != "default":
            X[int(k), 0] = v
    return _bits(W), _bits(X)


def _check_bw(c):
    W, X = _bw_inputs(c)
    keep = np.array(c["keep_blocks"], dtype=np.int32)
    form = bw.prune(W, DT, keep)
    Y, B = bw.gemm(form, keep, X, DT, DT, 256, c["alpha"])
    rows = c["rows"]
    assert (_vals(Y[rows]) == np.array(c["Y"])).all()
    assert (B[rows] == np.array(c["B"])).all()


def _check_ew(c):
    W, X = _bits(c["W"]), _bits(c["X"])
    M, K = W.shape
    form = ew.prune(W, DT, c["k"])
    Y, B = ew.spmm(form, M, K, X, DT, DT, c["alpha"])
    assert (_vals(Y) == np.array(c["Y"])).all()
    assert (B == np.array(c["B"])).all()


def _conv_inputs(c):
    Cin = c["Cin"]
    Wf = np.zeros((1, 9 * Cin))
    for tap, vals in c["taps"].items():
        Wf[0, int(tap) * Cin:(int(tap) + 1) * Cin] = vals
    X = np.array(c["pixels"]).reshape(1, 1, 2, Cin)
    return _bits(Wf), _bits(X)


def _check_conv(c, sparse):
    Wf, X = _conv_inputs(c)
    Y, B = conv.conv3x3(Wf, X, DT, DT, c["alpha"], sparse=sparse)
    key = "sp24" if sparse else "dense"
    assert (_vals(Y) == np.array(c[f"{key}_Y"])).all()
    assert (B == np.array(c[f"{key}_B"])).all()


def _check_all(fx):
    _check_dense(fx["dense_2x2"])
    _check_sp24(fx["sp24_row"])
    _check_tw(fx["tw_two_tiles"], False)
    _check_tw(fx["tw_two_tiles"], True)
    _check_bw(fx["bw_two_tiles"])
    _check_ew(fx["ew_rows"])
    _check_conv(fx["conv_1x2"], False)
    _check_conv(fx["conv_1x2"], True)


def test_hand_values_of_every_product_form(fx):
    _check_all(fx)


def test_fixture_discriminates(fx):
    """The fixture itself can tell the mistakes apart: a negative alpha, Y with
    cancellation (|Y| < B somewhere), and a bound over the unpruned weights that
    differs from the pruned one."""
    for key in ("dense_2x2", "sp24_row", "tw_two_tiles", "bw_two_tiles", "ew_rows", "conv_1x2"):
        assert fx[key]["alpha"] < 0
    d = fx["dense_2x2"]
    assert (np.abs(np.array(d["Y"])) < np.array(d["B"])).any()
    s = fx["sp24_row"]
    W, X = _bits(s["W"]), _bits(s["X"])
    assert (gemm.bound(W, X, DT, s["alpha"]) == np.array(s["B_unpruned"])).all()
    assert s["B_unpruned"] != s["B"]


@pytest.mark.parametrize("mistake", ["signed_alpha", "no_alpha", "squared_alpha"])
def test_planted_bound_mistakes_fail(fx, monkeypatch, mistake):
    """Each planted mistake in the one place the bound is computed must make at
    least one hand value fail."""
    def signed(Wd, Xd, alpha=1.0):
        return alpha * (np.abs(Wd) @ np.abs(Xd))

    def dropped(Wd, Xd, alpha=1.0):
        return np.abs(Wd) @ np.abs(Xd)

    def squared(Wd, Xd, alpha=1.0):
        return alpha * alpha * (np.abs(Wd) @ np.abs(Xd))

    plant = {"signed_alpha": signed, "no_alpha": dropped, "squared_alpha": squared}[mistake]
    monkeypatch.setattr(gemm, "bound_decoded", plant)
    with pytest.raises(AssertionError):
        _check_all(fx)


def test_planted_unpruned_bound_fails(fx):
    """The bound taken over the unpruned weights (the 2:4 case) misses the hand value."""
    s = fx["sp24_row"]
    W, X = _bits(s["W"]), _bits(s["X"])
    assert not (gemm.bound(W, X, DT, s["alpha"]) == np.array(s["B"])).all()


def test_within_bound_uses_the_bound_elementwise(fx):
    """within_bound accepts |Y - Y_ref| <= rel B elementwise and nothing more: on the
    2x2 fixture a perturbation of exactly rel B passes, one step (ulp) beyond fails,
    and where B == 0 only equality passes."""
    d = fx["dense_2x2"]
    B = np.array(d["B"])
    Y_ref = _bits(d["Y"])
    rel = 0.25
    ok = _vals(Y_ref) + rel * B                           # exact in bf16 here (dyadic, few bits)
    assert gemm.within_bound(_bits(ok), Y_ref, B, DT, rel).all()
    over = _vals(Y_ref) + rel * B * 1.25
    assert not gemm.within_bound(_bits(over), Y_ref, B, DT, rel).any()
    Z = np.zeros((1, 2))
    assert gemm.within_bound(_bits(Z), _bits(Z), Z, DT, rel).all()
    assert not gemm.within_bound(_bits([[2.0 ** -20, 0.0]]), _bits(Z), Z, DT, rel)[0, 0]
