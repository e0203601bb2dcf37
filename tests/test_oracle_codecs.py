"""Pins for the oracle's element codecs: format definitions, exhaustive
agreement with independent library casts, and hand-chosen boundary values."""
import numpy as np
import torch

from oracle import codecs


def test_fp16_decode_exhaustive_matches_numpy():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = codecs.decode(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_bf16_decode_exhaustive_matches_torch():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = codecs.decode(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_e4m3_decode_exhaustive_matches_torch():
    bits = np.arange(256, dtype=np.uint8)
    ours = codecs.decode(bits, "e4m3")
    ref = torch.from_numpy(bits.copy()).view(torch.float8_e4m3fn).double().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_e4m3_definition_points():
    d = lambda b: float(codecs.decode(np.array([b], np.uint8), "e4m3")[0])
    assert d(0x7E) == 448.0              # S.1111.110: largest finite
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert d(0x01) == 2.0 ** -9          # smallest subnormal
    assert d(0x08) == 2.0 ** -6          # smallest normal
    assert d(0x38) == 1.0                # exponent 7 = bias
    assert d(0xB8) == -1.0
    assert d(0x80) == 0.0 and np.signbit(d(0x80))


def test_round_ties_to_even_and_limits():
    # bf16 has 8 significant bits: 1 + 2**-8 is a tie between 1 and 1 + 2**-7.
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 1 + 2.0 ** -8 + 2.0 ** -30])
    assert list(codecs.round_to(x, "bf16")) == [1.0, 1 + 2.0 ** -6, -1.0, 1 + 2.0 ** -7]
    # fp16: 2049 is a tie between 2048 and 2050 -> 2048; 2051 -> 2052.
    assert list(codecs.round_to(np.array([2049.0, 2051.0]), "f16")) == [2048.0, 2052.0]
    # overflow: fp16 max 65504; 65520 rounds up to 2**16 -> inf.
    r = codecs.round_to(np.array([65504.0, 65519.0, 65520.0]), "f16")
    assert r[0] == 65504.0 and r[1] == 65504.0 and np.isinf(r[2])
    # e4m3 saturates
    assert list(codecs.round_to(np.array([464.0, 1e6, -1e6]), "e4m3")) == [448.0, 448.0, -448.0]
    # subnormals: fp16 smallest subnormal 2**-24; half of it ties to 0 (even).
    assert list(codecs.round_to(np.array([2.0 ** -25, 3 * 2.0 ** -25]), "f16")) == [0.0, 2.0 ** -23]


def test_encode_matches_library_rounding_on_random_values():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000)
    # fp16: numpy's double -> half conversion is an independent RNE implementation
    assert (codecs.encode(x, "f16") == x.astype(np.float16).view(np.uint16)).all()
    # bf16: torch rounds fp32 -> bf16; compare on values exactly representable in fp32
    x32 = x.astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x32.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (codecs.encode(x32, "bf16") == ref).all()


def test_decode_encode_roundtrip_exhaustive():
    for dt in ("f16", "bf16"):
        bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
        v = codecs.decode(bits, dt)
        fin = np.isfinite(v)
        assert (codecs.encode(v[fin], dt) == bits[fin]).all()
    bits = np.arange(256, dtype=np.uint8)
    v = codecs.decode(bits, "e4m3")
    fin = np.isfinite(v)
    assert (codecs.encode(v[fin], "e4m3") == bits[fin]).all()


def test_e4m3_encode_matches_torch_cast_inside_the_finite_range():
    """torch's fp32 -> float8_e4m3fn cast is an independent RNE implementation;
    compared on fp32 values within +-448 (where saturation plays no part),
    including the subnormal range and exact ties."""
    rng = np.random.default_rng(1)
    x = rng.uniform(-448, 448, 20000) * 2.0 ** rng.integers(-14, 1, 20000)
    ties = np.array([1.0625, 1.1875, 2.0 ** -9 * 1.5, 2.0 ** -9 * 0.5, -2.0 ** -9 * 2.5, 240.0 + 8.0])
    x = np.concatenate([x, ties]).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (codecs.encode(x, "e4m3") == ref).all()
