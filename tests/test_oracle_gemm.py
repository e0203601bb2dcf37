"""Pins for the oracle GEMM: identity, exact closed forms, brute-force triple
loops on tiny shapes, an independent library matmul, and planted mistakes."""
import numpy as np
import pytest
import torch

from oracle import codecs, gemm, sp24


def _bits(vals, dt):
    return codecs.encode(np.asarray(vals, dtype=np.float64), dt)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_identity_gives_rounded_pruned_w(dt):
    rng = np.random.default_rng(3)
    M, K = 20, 24
    W = _bits(rng.standard_normal((M, K)), dt)
    v, m = sp24.compress(W, dt)
    X = _bits(np.eye(K), dt)
    Y = gemm.gemm_sp24(v, m, K, X, dt, dt)
    assert (Y == sp24.prune(W, dt)).all()


def test_closed_form_powers_of_two():
    # W kept values are +-2**e, X small integers: every product and sum is exact,
    # so Y is the closed form sum_g (v0 x[k0] + v1 x[k1]) computed by hand below.
    M, K, N = 3, 8, 2
    Wf = np.array([[0, 2.0, 0, -4.0, 0.5, 0, 0.25, 0],
                   [1.0, 1.0, 0, 0, 0, 0, -8.0, 2.0],
                   [0, 0, 0, 0, 0, 0, 0, 0]])
    Xf = np.array([[1, 2], [3, -1], [5, 0], [-2, 7], [4, 4], [9, 9], [8, -8], [6, 1]], dtype=np.float64)
    expect = np.array([[2 * 3 - 4 * -2 + 0.5 * 4 + 0.25 * 8, 2 * -1 - 4 * 7 + 0.5 * 4 + 0.25 * -8],
                       [1 + 3 - 64 + 12, 2 - 1 + 64 + 2],
                       [0, 0]])
    W = _bits(Wf, "bf16")
    X = _bits(Xf, "bf16")
    v, m = sp24.compress(W, "bf16")
    Y = codecs.decode(gemm.gemm_sp24(v, m, K, X, "bf16", "bf16"), "bf16")
    assert (Y == expect).all()
    # alpha scales exactly by a power of two
    Y2 = codecs.decode(gemm.gemm_sp24(v, m, K, X, "bf16", "bf16", alpha=0.25), "bf16")
    assert (Y2 == expect * 0.25).all()


@pytest.mark.parametrize("dt,out_dt", [("f16", "f16"), ("bf16", "bf16"), ("e4m3", "bf16")])
def test_brute_force_triple_loop(dt, out_dt):
    rng = np.random.default_rng(5)
    M, K, N = 6, 8, 5
    if dt == "e4m3":
        W = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
        W[(W & 0x7F) == 0x7F] = 0x3A
        X = rng.integers(0, 256, size=(K, N)).astype(np.uint8)
        X[(X & 0x7F) == 0x7F] = 0x22
    else:
        W = _bits(rng.integers(-8, 9, size=(M, K)) / 4.0, dt)
        X = _bits(rng.integers(-8, 9, size=(K, N)) / 2.0, dt)
    alpha = 0.5
    v, m = sp24.compress(W, dt)
    Y = gemm.gemm_sp24(v, m, K, X, dt, out_dt, alpha=alpha)
    # brute force: decide the kept positions group by group, then sum in Python floats
    wv = codecs.decode(W, dt)
    xv = codecs.decode(X, dt)
    for i in range(M):
        for j in range(N):
            acc = 0.0
            for g in range(K // 4):
                mags = [abs(wv[i, 4 * g + p]) for p in range(4)]
                order = sorted(range(4), key=lambda p: (-mags[p], p))[:2]
                for p in order:
                    acc += wv[i, 4 * g + p] * xv[4 * g + p, j]
            ref = np.array([alpha * acc])
            # exact products/sums here (small dyadic values), so rounding is unambiguous
            assert Y[i, j] == codecs.encode(ref, out_dt)[0]


def test_matches_torch_float64_and_bound_holds():
    rng = np.random.default_rng(7)
    M, K, N = 37, 72, 29
    W = _bits(rng.standard_normal((M, K)), "bf16")
    X = _bits(rng.standard_normal((K, N)), "bf16")
    v, m = sp24.compress(W, "bf16")
    Wh = sp24.decompress(v, m, K)
    yt = (torch.from_numpy(codecs.decode(Wh, "bf16")) @ torch.from_numpy(codecs.decode(X, "bf16"))).numpy()
    Y = codecs.decode(gemm.gemm_sp24(v, m, K, X, "bf16", "bf16"), "bf16")
    B = gemm.bound(Wh, X, "bf16")
    assert (np.abs(Y - yt) <= 2.0 ** -8 * np.abs(yt) + 1e-30).all()   # one bf16 rounding
    assert (np.abs(Y - yt) <= 1e-2 * B).all()
    ok = gemm.within_bound(gemm.gemm_sp24(v, m, K, X, "bf16", "bf16"),
                           codecs.encode(yt, "bf16"), B, "bf16", 1e-2)
    assert ok.all()


def test_bound_detects_transposed_or_dropped_term():
    """Planted mistakes (transposed X, a dropped k term) break the bound check."""
    rng = np.random.default_rng(9)
    M, K, N = 16, 16, 16
    W = _bits(rng.standard_normal((M, K)), "f16")
    X = _bits(rng.standard_normal((K, N)), "f16")
    v, m = sp24.compress(W, "f16")
    Wh = sp24.decompress(v, m, K)
    good = gemm.gemm_sp24(v, m, K, X, "f16", "f16")
    B = gemm.bound(Wh, X, "f16")
    assert gemm.within_bound(good, good, B, "f16", 1e-2).all()
    bad_t = gemm.gemm_sp24(v, m, K, np.ascontiguousarray(X.T), "f16", "f16")
    assert not gemm.within_bound(bad_t, good, B, "f16", 1e-2).all()
    Wd = Wh.copy()
    Wd[:, -4:] = 0
    bad_d = gemm.gemm_dense(Wd, X, "f16", "f16")
    assert not gemm.within_bound(bad_d, good, B, "f16", 1e-2).all()


def test_rows_subset_equals_full():
    rng = np.random.default_rng(11)
    W = _bits(rng.standard_normal((40, 32)), "bf16")
    X = _bits(rng.standard_normal((32, 9)), "bf16")
    v, m = sp24.compress(W, "bf16")
    full = gemm.gemm_sp24(v, m, 32, X, "bf16", "bf16")
    rows = np.array([0, 5, 39])
    assert (gemm.gemm_sp24(v, m, 32, X, "bf16", "bf16", rows=rows) == full[rows]).all()
