"""The fused layer epilogue of the GEMM: bias, activation, output scaling.

A pruned fully connected layer or 1x1 convolution ("Accelerating Sparse DNNs
Based on Tiled GEMM", Abstract: the pruned layers run as GEMMs) produces
    Y[i, j] = round_out( y_scale * act( alpha * (W_hat . X)[i, j] + bias[i] ) )
with one bias per output feature i (a row of W and of Y), and the activation
applied before the layer's output is stored. Fusing this step into the GEMM
kernel follows the same page's "kernel fusion" (TL;DR). The output may be e4m3,
in which case y_scale is the reciprocal of the output tensor's quantisation
scale (a multiplier, applied before the one rounding).

Numerics: the product in fp64 through a library matmul; bias add, activation
and scaling in fp64; one rounding to the output type (ties to even; e4m3
saturates to +-448). GELU is the exact form x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)).
"""
from __future__ import annotations

import math

import numpy as np

from . import codecs, gemm, sp24

ACTS = ("none", "relu", "gelu")
# max |d act / dz|: 1 for the identity and ReLU; for GELU, Phi(z) + z phi(z)
# peaks at z = sqrt(2) with 0.92135 + 0.20755 = 1.1289
LIPSCHITZ = {"none": 1.0, "relu": 1.0, "gelu": 1.13}


def _erf(x: np.ndarray) -> np.ndarray:
    try:
        from scipy.special import erf
        return erf(x)
    except ImportError:  # pragma: no cover - scipy is present on both machines
        return np.vectorize(math.erf)(x)


def activation(z: np.ndarray, act: str) -> np.ndarray:
    """The activation in fp64."""
    z = np.asarray(z, dtype=np.float64)
    if act == "none":
        return z
    if act == "relu":
        return np.where(z > 0, z, 0.0)
    if act == "gelu":
        return 0.5 * z * (1.0 + _erf(z / math.sqrt(2.0)))
    raise ValueError(act)


def apply(acc: np.ndarray, bias, act: str, y_scale: float) -> np.ndarray:
    """y_scale * act(acc + bias[:, None]) in fp64 (acc already includes alpha)."""
    z = acc if bias is None else acc + np.asarray(bias, dtype=np.float64)[:, None]
    return y_scale * activation(z, act)


def gemm_sp24_ep(values, meta, K, X, dt, out_dt, alpha=1.0, bias=None, act="none", y_scale=1.0,
                 rows=None) -> np.ndarray:
    """Output bits of the 2:4 GEMM with the fused epilogue (optionally on a row subset)."""
    if rows is not None:
        values, meta = values[rows], meta[rows]
        bias = None if bias is None else np.asarray(bias)[rows]
    W_hat = sp24.decompress(values, meta, K)
    acc = gemm.dense_product(W_hat, X, dt, alpha)
    return codecs.encode(apply(acc, bias, act, y_scale), out_dt)


def gemm_dense_ep(W, X, dt, out_dt, alpha=1.0, bias=None, act="none", y_scale=1.0, rows=None) -> np.ndarray:
    """Output bits of the dense GEMM with the fused epilogue."""
    acc = gemm.dense_product(W, X, dt, alpha, rows)
    if rows is not None and bias is not None:
        bias = np.asarray(bias)[rows]
    return codecs.encode(apply(acc, bias, act, y_scale), out_dt)


def ulp(x: np.ndarray, dt: str) -> np.ndarray:
    """Spacing of dt's representable values at |x| (the subnormal spacing near 0)."""
    p, qmin_exp, _ = codecs._FORMATS[dt]
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.where(x > 0, x, 1.0))
    q = np.ldexp(1.0, np.maximum(e - p, qmin_exp))
    return np.where(x > 0, q, np.ldexp(1.0, qmin_exp))


def within_bound_ep(Y_bits, Y_ref_bits, B, out_dt: str, rel: float, act: str, y_scale: float) -> np.ndarray:
    """Elementwise check of an epilogue output against the reference.

    The accumulator may differ from the exact product by rel * B (B the
    |alpha| sum_k |w_ik x_kj| bound); the activation scales that by at most its
    Lipschitz constant and y_scale scales the rest; each side then rounds once
    to the output type, so one output ulp is allowed on top.
    """
    y = codecs.decode(Y_bits, out_dt)
    r = codecs.decode(Y_ref_bits, out_dt)
    d = np.abs(y - r)
    slack = LIPSCHITZ[act] * abs(y_scale) * rel * B + ulp(np.maximum(np.abs(y), np.abs(r)), out_dt)
    return (d <= slack) & np.isfinite(y)
