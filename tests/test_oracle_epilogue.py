"""Pins for the oracle's fused layer epilogue: a hand-derived fixture, standard
normal CDF table values for GELU, its reflection identity, output ulps, and
planted mistakes (bias after the activation, scale inside it, a dropped bias)."""
import json
import math
import os

import numpy as np
import pytest

from oracle import codecs, epilogue, gemm, sp24

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "epilogue_hand.json")


def _fixture():
    with open(GOLDEN) as f:
        g = json.load(f)
    W = codecs.encode(np.array(g["W"]), g["dtype"])
    X = codecs.encode(np.eye(g["K"]), g["dtype"])
    return g, W, X


@pytest.mark.parametrize("act", ["none", "relu"])
def test_hand_fixture(act):
    g, W, X = _fixture()
    v, m = sp24.compress(W, g["dtype"])
    Y = epilogue.gemm_sp24_ep(v, m, g["K"], X, g["dtype"], g["out_dtype"], g["alpha"], np.array(g["bias"]),
                              act, g["y_scale"])
    assert Y.tolist() == g[f"codes_{act}"]
    Yd = epilogue.gemm_dense_ep(W, X, g["dtype"], g["out_dtype"], g["alpha"], np.array(g["bias"]), act,
                                g["y_scale"])
    assert Yd.tolist() == g[f"codes_{act}"]


def test_planted_mistakes_fail_the_fixture():
    g, W, X = _fixture()
    acc = gemm.dense_product(W, X, g["dtype"])
    b = np.array(g["bias"])[:, None]
    s = g["y_scale"]
    want = np.array(g["codes_relu"])
    bias_after = codecs.encode(s * (np.maximum(acc, 0) + b), "e4m3")           # bias after the activation
    assert not np.array_equal(bias_after, want)
    scale_inside = codecs.encode(np.maximum(s * acc + b, 0), "e4m3")          # scale before bias / act
    assert not np.array_equal(scale_inside, want)
    no_bias = codecs.encode(s * np.maximum(acc, 0), "e4m3")
    assert not np.array_equal(no_bias, want)


def test_gelu_is_x_times_the_normal_cdf():
    # standard normal CDF table values Phi(x)
    table = {0.5: 0.691462461274013, 1.0: 0.841344746068543, 1.5: 0.933192798731142,
             2.0: 0.977249868051821, 3.0: 0.998650101968370}
    for x, phi in table.items():
        assert abs(epilogue.activation(np.array([x]), "gelu")[0] - x * phi) < 1e-14
        assert abs(epilogue.activation(np.array([-x]), "gelu")[0] - (-x) * (1 - phi)) < 1e-14
    assert epilogue.activation(np.array([0.0]), "gelu")[0] == 0.0
    # far tails: GELU(x) -> x for large x, -> 0 for very negative x
    assert epilogue.activation(np.array([40.0]), "gelu")[0] == 40.0
    assert abs(epilogue.activation(np.array([-40.0]), "gelu")[0]) < 1e-300


def test_gelu_reflection_identity():
    # Phi(-x) = 1 - Phi(x)  =>  GELU(-x) = GELU(x) - x
    x = np.random.default_rng(3).standard_normal(1000) * 3
    lhs = epilogue.activation(-x, "gelu")
    rhs = epilogue.activation(x, "gelu") - x
    assert np.allclose(lhs, rhs, rtol=0, atol=1e-13)


def test_gelu_lipschitz_constant():
    z = np.linspace(-8, 8, 160001)
    d = np.diff(epilogue.activation(z, "gelu")) / np.diff(z)
    assert d.max() <= epilogue.LIPSCHITZ["gelu"] and d.max() > 1.12


def test_relu_and_identity():
    z = np.array([-2.0, -0.0, 0.0, 1e-30, 3.5])
    assert epilogue.activation(z, "relu").tolist() == [0.0, 0.0, 0.0, 1e-30, 3.5]
    assert epilogue.activation(z, "none").tolist() == z.tolist()


def test_e4m3_output_saturates_and_rounds_to_even():
    acc = np.array([[1000.0, -1000.0, 1.5 * 2.0 ** -9, 1.0625, 1.1875]])
    Y = codecs.encode(epilogue.apply(acc, None, "none", 1.0), "e4m3")
    # 448 = 0x7E; 1.5 * 2^-9 ties between 1 and 2 subnormal steps -> 2 (even) = 0x02;
    # 1.0625 ties between 1 and 1.125 -> 1 (0x38); 1.1875 -> 1.25 (0x3A)
    assert Y.tolist() == [[0x7E, 0xFE, 0x02, 0x38, 0x3A]]


def test_ulp_values():
    assert epilogue.ulp(np.array([1.0]), "bf16")[0] == 2.0 ** -7
    assert epilogue.ulp(np.array([1.0]), "f16")[0] == 2.0 ** -10
    assert epilogue.ulp(np.array([1.0]), "e4m3")[0] == 2.0 ** -3
    assert epilogue.ulp(np.array([448.0]), "e4m3")[0] == 32.0
    assert epilogue.ulp(np.array([0.0]), "e4m3")[0] == 2.0 ** -9
    assert epilogue.ulp(np.array([-3.0]), "f16")[0] == 2.0 ** -9


@pytest.mark.parametrize("out_dt", ["bf16", "e4m3"])
@pytest.mark.parametrize("act", ["relu", "gelu"])
def test_checker_accepts_reference_and_rejects_a_dropped_bias(out_dt, act):
    rng = np.random.default_rng(5)
    M, K, N = 24, 64, 16
    W = codecs.encode(rng.standard_normal((M, K)) * 0.1, "bf16")
    X = codecs.encode(rng.standard_normal((K, N)), "bf16")
    bias = rng.standard_normal(M).astype(np.float32).astype(np.float64)
    v, m = sp24.compress(W, "bf16")
    ys = 4.0 if out_dt == "e4m3" else 1.0
    ref = epilogue.gemm_sp24_ep(v, m, K, X, "bf16", out_dt, 1.0, bias, act, ys)
    B = gemm.bound(sp24.decompress(v, m, K), X, "bf16")
    assert epilogue.within_bound_ep(ref, ref, B, out_dt, 1e-2, act, ys).all()
    wrong = epilogue.gemm_sp24_ep(v, m, K, X, "bf16", out_dt, 1.0, None, act, ys)
    assert not epilogue.within_bound_ep(wrong, ref, B, out_dt, 1e-2, act, ys).all()


def test_rows_subset_equals_full():
    rng = np.random.default_rng(7)
    W = codecs.encode(rng.standard_normal((40, 32)), "f16")
    X = codecs.encode(rng.standard_normal((32, 8)), "f16")
    bias = rng.standard_normal(40)
    v, m = sp24.compress(W, "f16")
    full = epilogue.gemm_sp24_ep(v, m, 32, X, "f16", "f16", 0.5, bias, "gelu", 2.0)
    rows = np.array([0, 7, 39])
    sub = epilogue.gemm_sp24_ep(v, m, 32, X, "f16", "f16", 0.5, bias, "gelu", 2.0, rows=rows)
    assert np.array_equal(sub, full[rows])
    assert math.isfinite(float(codecs.decode(full, "f16").sum()))
