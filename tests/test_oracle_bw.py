"""Pins for the oracle's block-wise sparsity: a hand fixture with exact block
scores and a tie, brute force over all block subsets, the masked-dense GEMM
identity, the limits (all blocks kept, none kept) and planted mistakes."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import bw, codecs, gemm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "bw_hand.json")


def _fixture_W(g):
    vals = np.array(g["block_values"])
    cols = np.repeat(vals, 64) * np.where(np.arange(g["K"]) % 2 == 0, 1.0, -1.0)
    return codecs.encode(np.tile(cols, (128, 1)), g["dtype"])


def test_hand_fixture_scores_and_selection():
    with open(GOLDEN) as f:
        g = json.load(f)
    W = _fixture_W(g)
    assert bw.block_scores(W, g["dtype"])[0].tolist() == g["scores"]
    for n in (1, 2, 3):
        form = bw.prune(W, g["dtype"], np.array([n]))
        assert form["indices"].tolist() == g[f"keep_{n}"]
        # the packed tile holds exactly the kept blocks' columns
        cols = np.concatenate([np.arange(64 * b, 64 * b + 64) for b in g[f"keep_{n}"]])
        assert np.array_equal(bw.unpack_tile(form, np.array([n]), 0), W[:, cols])


def test_planted_mistakes_fail_the_fixture():
    with open(GOLDEN) as f:
        g = json.load(f)
    s = np.array(g["scores"])
    # ties to the higher block index
    order_hi = sorted(range(4), key=lambda b: (-s[b], -b))[:1]
    assert order_hi != g["keep_1"]
    # scoring by the largest |w| of a block instead of the sum cannot separate equal-peak blocks
    peak = np.array(g["block_values"])
    order_peak = sorted(range(4), key=lambda b: (-peak[b], b))[:3]
    assert sorted(order_peak) == g["keep_3"]          # agrees here ...
    W = _fixture_W(g)
    Wb = codecs.decode(W, "bf16").copy()
    Wb[:, 64:128] = 0
    Wb[0, 64] = 3.0                                    # block 1: same peak, far smaller sum
    form = bw.prune(codecs.encode(Wb, "bf16"), "bf16", np.array([2]))
    assert form["indices"].tolist() == [2, 3]          # ... but not here: the sum decides


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_brute_force_over_block_subsets(seed):
    rng = np.random.default_rng(seed)
    W = codecs.encode(rng.standard_normal((200, 384)) * rng.uniform(0.1, 2.0, size=(1, 384)), "bf16")
    keep = np.array([2, 4])
    form = bw.prune(W, "bf16", keep)
    Wd = np.abs(codecs.decode(W, "bf16"))
    for t, n in enumerate(keep):
        rows = Wd[128 * t:min(200, 128 * (t + 1))]
        sums = [rows[:, 64 * b:64 * (b + 1)].sum() for b in range(6)]       # fp64, independent order
        best = max(itertools.combinations(range(6), int(n)), key=lambda c: (sum(sums[b] for b in c), [-b for b in c]))
        got = form["indices"][form["offsets"][t]:form["offsets"][t + 1]].tolist()
        assert got == sorted(best)


def test_gemm_equals_masked_dense_and_limits():
    rng = np.random.default_rng(7)
    M, K, N = 300, 256, 24
    W = codecs.encode(rng.standard_normal((M, K)), "bf16")
    X = codecs.encode(rng.standard_normal((K, N)), "bf16")
    keep = np.array([1, 4, 0])
    form = bw.prune(W, "bf16", keep)
    Y, B = bw.gemm(form, keep, X, "bf16", "bf16", M)
    Wm = bw.masked_dense(W, form, keep)
    Y_ref = gemm.gemm_dense(Wm, X, "bf16", "bf16")
    assert gemm.within_bound(Y, Y_ref, B, "bf16", 1e-6).all()
    assert (codecs.decode(Y[256:], "bf16") == 0).all()                      # tile 2 keeps nothing
    # every block kept: the dense product
    full = bw.prune(W, "bf16", np.array([4, 4, 4]))
    Yf, _ = bw.gemm(full, np.array([4, 4, 4]), X, "bf16", "bf16", M)
    assert np.array_equal(Yf, gemm.gemm_dense(W, X, "bf16", "bf16"))


def test_layout_offsets_and_schedule():
    rng = np.random.default_rng(9)
    W = codecs.encode(rng.standard_normal((384, 320)), "f16")
    keep = np.array([3, 0, 5])
    form = bw.prune(W, "f16", keep)
    assert form["offsets"].tolist() == [0, 3, 3, 8]
    assert form["packed"].size == 128 * 64 * 8
    # schedule: tiles by kept columns descending (t, L, P, Q)
    assert form["schedule_table"].reshape(-1, 4).tolist() == [[2, 320, 192, 3], [0, 192, 0, 0], [1, 0, 192, 3]]
