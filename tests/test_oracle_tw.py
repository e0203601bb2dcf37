"""Pins for the oracle's tile-wise (TW) and tile-vector-wise (TVW) steps:
hand-derived fixture, brute force over all subsets on tiny K, reductions to
the dense GEMM (L = K) and to zeros (L = 0), layout invariants, TVW = 2:4
applied to the packed tile, and a planted mistake."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import codecs, gemm, sp24, tw


def _hand(golden_dir):
    with open(os.path.join(golden_dir, "tw_hand.json")) as f:
        g = json.load(f)
    K = g["K"]
    Wf = np.zeros((128, K))
    Wf[0] = g["row0"]
    Wf[1] = g["row1"]
    return g, codecs.encode(Wf, "bf16")


def _check_hand(golden_dir):
    g, W = _hand(golden_dir)
    s = tw.scores(W, "bf16")
    assert list(s[0]) == g["scores"]
    for L, kept in g["kept"].items():
        assert list(tw.select(s[0], int(L))) == kept


def test_hand_fixture(golden_dir):
    _check_hand(golden_dir)


def test_planted_mistake_is_caught(golden_dir, monkeypatch):
    def ties_to_higher(s_t, L):
        K = s_t.shape[0]
        order = np.lexsort((-np.arange(K), -s_t.astype(np.float64)))
        return np.sort(order[:L]).astype(np.int32)

    with monkeypatch.context() as m:
        m.setattr(tw, "select", ties_to_higher)
        with pytest.raises(AssertionError):
            _check_hand(golden_dir)


def test_scores_are_sequential_fp32():
    rng = np.random.default_rng(2)
    W = codecs.encode(rng.standard_normal((130, 12)) * 10.0 ** rng.integers(-3, 4, (130, 12)), "bf16")
    s = tw.scores(W, "bf16")
    a = np.abs(codecs.decode(W, "bf16"))
    for t, (r0, r1) in enumerate([(0, 128), (128, 130)]):
        for k in range(12):
            acc = np.float32(0)
            for i in range(r0, r1):
                acc = np.float32(acc + np.float32(a[i, k]))
            assert s[t, k] == acc


def test_select_brute_force_all_subsets():
    rng = np.random.default_rng(4)
    K = 8
    for trial in range(30):
        s_t = rng.integers(0, 4, K).astype(np.float32)     # many ties
        for L in range(K + 1):
            best = None
            for sub in itertools.combinations(range(K), L):
                # the chosen set maximises the sorted score vector, then prefers
                # lower indices (lexicographically smallest index tuple)
                key = (tuple(sorted((-s_t[k] for k in sub))), sub)
                if best is None or key < best[0]:
                    best = (key, sub)
            assert tuple(tw.select(s_t, L)) == best[1]


def _rand_w(M, K, seed, dt="bf16"):
    rng = np.random.default_rng(seed)
    return codecs.encode(rng.standard_normal((M, K)) * 0.02, dt)


@pytest.mark.parametrize("tvw", [False, True])
def test_layout_invariants_and_unpack(tvw):
    M, K = 300, 200
    W = _rand_w(M, K, 6)
    keep = np.array([8, 0, 200], dtype=np.int32) if tvw else np.array([7, 0, 200], dtype=np.int32)
    f = tw.prune(W, "bf16", keep, tvw)
    off = f["offsets"]
    assert off[0] == 0 and list(np.diff(off)) == list(keep) and off[-1] == keep.sum()
    assert f["indices"].size == keep.sum()
    for t in range(3):
        idx = f["indices"][off[t]:off[t + 1]]
        assert len(idx) == keep[t] and (np.diff(idx) > 0).all() and (idx >= 0).all() and (idx < K).all()
        blk = tw.unpack_tile(f, keep, t, tvw, "bf16")
        dense = tw.gathered_tile(W, t, idx)
        if tvw:
            assert (blk == sp24.prune(dense, "bf16")).all() if keep[t] else blk.size == 0
        else:
            assert (blk == dense).all()
    assert list(f["schedule"]) == [2, 0, 1]
    R = tw.padded(keep.astype(np.int64))
    P = [0, R[0], R[0] + R[1]]
    Q = [0, (R[0] + 127) // 128, (R[0] + 127) // 128 + (R[1] + 127) // 128]
    assert list(f["schedule_table"]) == [2, keep[2], P[2], Q[2], 0, keep[0], P[0], Q[0], 1, keep[1], P[1], Q[1]]
    R = tw.padded(keep.astype(np.int64))
    assert f["packed"].size == 128 * R.sum() // (2 if tvw else 1)


def test_tvw_equals_sp24_on_packed_tile():
    M, K = 128, 96
    W = _rand_w(M, K, 8)
    keep = np.array([64], dtype=np.int32)
    f = tw.prune(W, "bf16", keep, True)
    idx = f["indices"]
    v, m = sp24.compress(tw.gathered_tile(W, 0, idx), "bf16")
    packed = f["packed"].reshape(1, 128, 32)[0]            # one 64-column chunk
    assert (packed == v[:, :32]).all()
    assert (f["meta"].reshape(128, 8) == m[:, :8]).all()
    assert (f["meta_hw"] == sp24.meta_hw_from_canonical(m[:, :8], 128, 64, "bf16")).all()


def test_full_keep_reduces_to_dense_and_empty_gives_zero():
    M, K, N = 256, 64, 24
    W = _rand_w(M, K, 10)
    X = codecs.encode(np.random.default_rng(11).standard_normal((K, N)), "bf16")
    keep = np.array([K, 0], dtype=np.int32)
    f = tw.prune(W, "bf16", keep, False)
    Y, B = tw.gemm(f, keep, X, "bf16", "bf16", M, False)
    Yd = gemm.gemm_dense(W[:128], X, "bf16", "bf16")
    assert (Y[:128] == Yd).all()
    assert (Y[128:] == 0).all() and (B[128:] == 0).all()
    # TVW with full keep reduces to the 2:4 GEMM
    f2 = tw.prune(W, "bf16", keep, True)
    Y2, _ = tw.gemm(f2, keep, X, "bf16", "bf16", M, True)
    v, m = sp24.compress(W[:128], "bf16")
    assert (Y2[:128] == gemm.gemm_sp24(v, m, K, X, "bf16", "bf16")).all()


def test_tw_equals_masked_dense_within_bound():
    M, K, N = 256, 128, 16
    W = _rand_w(M, K, 12)
    X = codecs.encode(np.random.default_rng(13).standard_normal((K, N)), "bf16")
    keep = np.array([40, 100], dtype=np.int32)
    f = tw.prune(W, "bf16", keep, False)
    Y, B = tw.gemm(f, keep, X, "bf16", "bf16", M, False)
    masked = np.zeros_like(W)
    for t in range(2):
        idx = f["indices"][f["offsets"][t]:f["offsets"][t + 1]]
        masked[t * 128:(t + 1) * 128, idx] = W[t * 128:(t + 1) * 128, idx]
    Yd = gemm.gemm_dense(masked, X, "bf16", "bf16")
    assert gemm.within_bound(Y, Yd, B, "bf16", 1e-2).all()
