"""Pins for the oracle's 2:4 prune / compress / decompress.

The pages define the pattern (two zeros in every contiguous group of four,
stored as values plus position metadata); the criterion (largest magnitudes),
tie rule and layouts are the readings stated in the design notes. Pins:
hand-derived fixtures, brute force over all six masks, the four invariants,
exhaustive e4m3 magnitude patterns, and planted mistakes that must be caught.
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import codecs, sp24

VALID_NIBBLES = {0x4, 0x8, 0xC, 0x9, 0xD, 0xE}


def _f16_bits(vals):
    return np.array(vals, dtype=np.float64).astype(np.float16).view(np.uint16)


def test_hand_fixture(golden_dir):
    _check_hand_fixture(golden_dir)


def _check_hand_fixture(golden_dir):
    with open(os.path.join(golden_dir, "sp24_hand_fp16.json")) as f:
        g = json.load(f)
    K = g["K"]
    W = np.stack([_f16_bits(r["w"]) for r in g["rows"]])
    values, meta = sp24.compress(W, "f16")
    Kp = sp24.padded_k(K)
    assert values.shape == (len(g["rows"]), Kp // 2) and meta.shape == (len(g["rows"]), Kp // 8)
    for i, r in enumerate(g["rows"]):
        assert list(values[i, :K // 2]) == list(_f16_bits(r["values"]))     # bits, incl. -0.0
        assert list(meta[i, :K // 8]) == r["meta_bytes"]
        n = sp24.nibbles(meta[i:i + 1], K // 4)[0]
        assert list(n) == r["nibbles"]
        j0, j1 = sp24.prune_positions(W[i:i + 1], "f16")
        assert [[a, b] for a, b in zip(j0[0], j1[0])] == r["kept_positions"]
        # padding past K: value 0, nibble 0x4
        assert (values[i, K // 2:] == 0).all()
        assert (meta[i, K // 8:] == 0x44).all()


def _brute_force_keep(mags):
    """Among the six 2-of-4 masks pick the one the rule selects, by enumeration:
    maximise the sorted kept magnitudes, then prefer lower positions."""
    best = None
    for pair in itertools.combinations(range(4), 2):
        kept = sorted((mags[p] for p in pair), reverse=True)
        dropped = [mags[p] for p in range(4) if p not in pair]
        # valid iff every kept magnitude >= every dropped one
        if min(kept) < max(dropped):
            continue
        # among valid masks, ties go to lower positions: lexicographically smallest pair
        key = (tuple(-m for m in kept), pair)
        if best is None or key < best[0]:
            best = (key, pair)
    return best[1]


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3"])
def test_brute_force_small_random(dt):
    rng = np.random.default_rng(1)
    # small integer-ish magnitudes to produce many ties
    if dt == "e4m3":
        W = rng.integers(0, 256, size=(64, 32)).astype(np.uint8)
        W[(W & 0x7F) == 0x7F] = 0x10          # finite inputs only
    else:
        vals = rng.integers(-3, 4, size=(64, 32)).astype(np.float64) * 0.5
        W = codecs.encode(vals, dt)
    j0, j1 = sp24.prune_positions(W, dt)
    mags = sp24.magnitude_key(W, dt)
    for i in range(W.shape[0]):
        for g in range(W.shape[1] // 4):
            assert (j0[i, g], j1[i, g]) == _brute_force_keep(list(mags[i, 4 * g:4 * g + 4]))


def test_e4m3_all_magnitude_pairs_exhaustive():
    # every ordered choice of magnitudes for two slots against fixed others
    codes = np.arange(0, 0x7F, dtype=np.uint8)              # all finite positive codes
    a, b = np.meshgrid(codes, codes, indexing="ij")
    n = a.size
    W = np.zeros((n, 4), dtype=np.uint8)
    W[:, 0] = a.reshape(-1)
    W[:, 1] = 0x38                                          # 1.0
    W[:, 2] = b.reshape(-1) | 0x80                          # negative values
    W[:, 3] = 0x30                                          # 0.5
    j0, j1 = sp24.prune_positions(W, "e4m3")
    dec = np.abs(codecs.decode(W, "e4m3"))
    for r in range(0, n, 97):                               # a spread sample of the 16129 rows
        assert (j0[r, 0], j1[r, 0]) == _brute_force_keep(list(dec[r]))
    # and the full set through the invariants
    kept = np.sort(np.stack([np.take_along_axis(dec, j0, 1)[:, 0], np.take_along_axis(dec, j1, 1)[:, 0]], 1), 1)
    mask = np.ones((n, 4), bool)
    mask[np.arange(n), j0[:, 0]] = False
    mask[np.arange(n), j1[:, 0]] = False
    dropped = np.where(mask, dec, -1).max(1)
    assert (kept[:, 0] >= dropped).all()


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("shape", [(5, 4), (7, 36), (130, 260), (3, 300)])
def test_invariants(dt, shape):
    rng = np.random.default_rng(["f16", "bf16", "e4m3"].index(dt) * 1000 + shape[0] * 7 + shape[1])
    M, K = shape
    if dt == "e4m3":
        W = rng.integers(0, 256, size=shape).astype(np.uint8)
        W[(W & 0x7F) == 0x7F] = 0x01
    else:
        W = codecs.encode(rng.standard_normal(shape), dt)
    values, meta = sp24.compress(W, dt)
    n = sp24.nibbles(meta, K // 4)
    # 1. exactly two distinct positions per group
    assert set(np.unique(n)) <= VALID_NIBBLES
    # 2. decompress(compress(W)) == prune(W) bit for bit, and has 2 zeros per group
    Wh = sp24.decompress(values, meta, K)
    assert (Wh == sp24.prune(W, dt)).all()
    kept_mask = np.zeros((M, K // 4, 4), bool)
    j0, j1 = n & 3, (n >> 2) & 3
    np.put_along_axis(kept_mask, j0[..., None].astype(np.int64), True, -1)
    np.put_along_axis(kept_mask, j1[..., None].astype(np.int64), True, -1)
    assert (kept_mask.sum(-1) == 2).all()
    assert (np.where(kept_mask.reshape(M, K), 0, Wh) == 0).all()
    # kept entries are W's own bits
    assert (np.where(kept_mask.reshape(M, K), Wh, 0) == np.where(kept_mask.reshape(M, K), W, 0)).all()
    # 3. smaller kept magnitude >= larger dropped magnitude; ties resolved to lower index
    mag = sp24.magnitude_key(W, dt).reshape(M, K // 4, 4)
    kept_min = np.where(kept_mask, mag, 1 << 20).min(-1)
    drop_max = np.where(kept_mask, -1, mag).max(-1)
    assert (kept_min >= drop_max).all()
    for i, g in zip(*np.nonzero(kept_min == drop_max)):
        tie = mag[i, g] == kept_min[i, g]
        kpos = [p for p in range(4) if kept_mask[i, g, p] and tie[p]]
        dpos = [p for p in range(4) if (not kept_mask[i, g, p]) and tie[p]]
        assert max(kpos) < min(dpos)
    # 4. the hardware-ordered metadata is a permutation of the canonical nibbles
    hw = sp24.meta_hw_from_canonical(meta, M, K, dt)
    assert hw.size == sp24.meta_hw_size(M, K, dt)
    assert (_canonical_from_hw(hw, M, K, dt)[:, :meta.shape[1]] == meta).all()


def _canonical_from_hw(hw, M, K, dt):
    """Independent inverse of the operand layout: rebuild canonical bytes row by row."""
    MB = (M + 127) // 128
    if dt == "e4m3":
        KB = (K + 127) // 128
        b = hw.reshape(MB, KB, 128, 16)
        out = np.zeros((MB * 128, KB * 16), np.uint8)
        for mb in range(MB):
            for kb in range(KB):
                out[mb * 128:(mb + 1) * 128, kb * 16:(kb + 1) * 16] = b[mb, kb]
        return out[:M]
    KB = (K + 63) // 64
    w = hw.view("<u4").reshape(MB, KB, 128, 4)
    out = np.zeros((MB * 128, KB * 2), np.uint32)
    for mb in range(MB):
        for kb in range(KB):
            for j in range(2):
                col = w[mb, kb, :, 2 * j]
                assert (w[mb, kb, :, 2 * j + 1] == 0).all()
                for r in range(128):
                    lo, hi = int(col[r]) & 0xFFFF, int(col[r]) >> 16
                    low_row = r & ~8
                    up_row = r | 8
                    if r & 8 == 0:    # groups 0..3 of rows r (low) and r + 8 (high)
                        out[mb * 128 + low_row, 2 * kb + j] |= lo
                        out[mb * 128 + up_row, 2 * kb + j] |= hi
                    else:             # groups 4..7 of rows r - 8 (low) and r (high)
                        out[mb * 128 + low_row, 2 * kb + j] |= lo << 16
                        out[mb * 128 + up_row, 2 * kb + j] |= hi << 16
    return out.view(np.uint8).reshape(MB * 128, -1)[:M]


def test_all_equal_and_signed_zero_groups():
    W = _f16_bits([[0.0, -0.0, 0.0, -0.0, 2, 2, 2, 2, -2, 2, -2, 2]])
    values, meta = sp24.compress(W, "f16")
    assert list(sp24.nibbles(meta, 3)[0]) == [4, 4, 4]
    assert list(values[0, :6]) == list(_f16_bits([0.0, -0.0, 2, 2, -2, 2]))


def test_k_not_multiple_of_four_rejected():
    with pytest.raises(ValueError):
        sp24.prune_positions(np.zeros((2, 6), np.uint16), "f16")


def test_planted_mistakes_are_caught(monkeypatch, golden_dir):
    """Plausible mistakes planted in the oracle must fail the hand fixture."""
    def tie_to_higher(bits, dt):
        M, K = bits.shape
        key = sp24.magnitude_key(bits, dt).reshape(M, K // 4, 4)
        order = 3 - np.argsort(-key[..., ::-1], axis=-1, kind="stable")
        top = np.sort(order[..., :2], axis=-1)
        return top[..., 0], top[..., 1]

    def signed_compare(bits, dt):          # forgets to clear the sign bit
        return bits.astype(np.int64).astype(np.int16 if dt != "e4m3" else np.int8).astype(np.int64)

    with monkeypatch.context() as m:
        m.setattr(sp24, "prune_positions", tie_to_higher)
        with pytest.raises(AssertionError):
            _check_hand_fixture(golden_dir)
    with monkeypatch.context() as m:
        m.setattr(sp24, "magnitude_key", signed_compare)
        with pytest.raises(AssertionError):
            _check_hand_fixture(golden_dir)
    _check_hand_fixture(golden_dir)
