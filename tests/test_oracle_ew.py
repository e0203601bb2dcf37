"""Pins for the oracle's element-wise (unstructured) pruning and SpMM: a
hand fixture with ties, the selection invariants on random rows, the product
against the dense product of the decompressed matrix, the limits, and a planted
signed-compare mistake."""
import json
import os

import numpy as np
import pytest

from oracle import codecs, ew, gemm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ew_hand.json")


def test_hand_fixture():
    with open(GOLDEN) as f:
        g = json.load(f)
    W = codecs.encode(np.array([g["row"]]), g["dtype"])
    for k in (1, 3, 5, 7):
        form = ew.prune(W, g["dtype"], k)
        assert form["col_idx"].tolist() == g[f"keep_{k}"]
        assert form["row_ptr"].tolist() == [0, k]
        assert np.array_equal(form["vals"], W[0, g[f"keep_{k}"]])      # bits copied, signs kept


def test_planted_signed_compare_fails():
    with open(GOLDEN) as f:
        g = json.load(f)
    row = np.array(g["row"])
    signed = sorted(np.argsort(-row, kind="stable")[:3].tolist())     # compares signed values
    assert signed != g["keep_3"]


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_selection_invariants(dt):
    rng = np.random.default_rng(3)
    W = codecs.encode(np.round(rng.standard_normal((40, 96)) * 4) / 4, dt)   # many ties
    k = 10
    form = ew.prune(W, dt, k)
    mag = W.astype(np.int64) & 0x7FFF
    cols = form["col_idx"].reshape(40, k)
    for i in range(40):
        kept = set(cols[i].tolist())
        assert len(kept) == k and list(cols[i]) == sorted(cols[i])
        dropped = [c for c in range(96) if c not in kept]
        lo = min(mag[i, c] for c in kept)
        hi = max(mag[i, c] for c in dropped)
        assert lo >= hi                                            # nothing dropped is larger
        for c in dropped:                                          # at the threshold, lower index kept
            if mag[i, c] == lo:
                assert all(kc < c for kc in kept if mag[i, kc] == lo)


def test_spmm_matches_dense_product_and_limits():
    rng = np.random.default_rng(5)
    M, K, N = 48, 128, 20
    W = codecs.encode(rng.standard_normal((M, K)), "bf16")
    X = codecs.encode(rng.standard_normal((K, N)), "bf16")
    form = ew.prune(W, "bf16", 13)
    Y, B = ew.spmm(form, M, K, X, "bf16", "bf16", alpha=0.5)
    Wd = ew.decompress(form, M, K)
    assert ((Wd != 0).sum(axis=1) <= 13).all()
    Y_ref = gemm.gemm_dense(Wd, X, "bf16", "bf16", 0.5)
    assert gemm.within_bound(Y, Y_ref, gemm.bound(Wd, X, "bf16", 0.5), "bf16", 1e-9).all()
    rows = np.array([0, 17, 47])
    Yr, _ = ew.spmm(form, M, K, X, "bf16", "bf16", alpha=0.5, rows=rows)
    assert np.array_equal(Yr, Y[rows])
    full = ew.prune(W, "bf16", K)
    assert np.array_equal(ew.decompress(full, M, K), W)
    Yf, _ = ew.spmm(full, M, K, X, "bf16", "bf16")
    assert gemm.within_bound(Yf, gemm.gemm_dense(W, X, "bf16", "bf16"), gemm.bound(W, X, "bf16"), "bf16", 1e-9).all()
    Y0, _ = ew.spmm(ew.prune(W, "bf16", 0), M, K, X, "bf16", "bf16")
    assert (codecs.decode(Y0, "bf16") == 0).all()
