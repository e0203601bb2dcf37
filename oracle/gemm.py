"""The GEMM Y = alpha * W_hat . X and its elementwise error bound.

W_hat is the decompressed (pruned) weight matrix: "Accelerating Sparse Deep
Neural Networks", Abstract (the sparse tensor core computes the product of the
2:4 matrix with a dense operand, skipping the zero half); "Accelerating Sparse
DNNs Based on Tiled GEMM", Abstract (pruned fully connected / convolution layers
as GEMM).

Numerics: products and sums in fp64 through a library matmul (a step, no
reordering beyond what the definition states), one multiply by alpha in fp64,
one rounding to the output type (ties to even). The pages fix no precision.
The error bound B_ij = |alpha| * sum_k |w_ik x_kj| is computed the same way.
"""
from __future__ import annotations

import numpy as np

from . import codecs, sp24


def dense_product(W: np.ndarray, X: np.ndarray, dt: str, alpha: float = 1.0,
                  rows=None) -> np.ndarray:
    """alpha * decode(W) . decode(X) in fp64 (W M x K bits, X K x N bits)."""
    Wd = codecs.decode(W if rows is None else W[rows], dt)
    Xd = codecs.decode(X, dt)
    return alpha * (Wd @ Xd)


def bound_decoded(Wd: np.ndarray, Xd: np.ndarray, alpha: float = 1.0) -> np.ndarray:
    """B_ij = |alpha| * sum_k |w_ik| |x_kj| in fp64 from decoded values: the scale of
    the elementwise tolerance |Y - Y_ref| <= rel * B. Every product form of the
    oracle (2:4, dense, tile-wise, block-wise, element-wise, convolution) takes its
    bound from here, over the weights it actually multiplies (the pruned ones)."""
    return abs(alpha) * (np.abs(Wd) @ np.abs(Xd))


def bound(W: np.ndarray, X: np.ndarray, dt: str, alpha: float = 1.0, rows=None) -> np.ndarray:
    """|alpha| * sum_k |w_ik| |x_kj| in fp64 (W and X as stored bits)."""
    return bound_decoded(codecs.decode(W if rows is None else W[rows], dt), codecs.decode(X, dt), alpha)


def gemm_dense(W: np.ndarray, X: np.ndarray, dt: str, out_dt: str, alpha: float = 1.0,
               rows=None) -> np.ndarray:
    """Y = round_out(alpha * W . X) as output-type bits."""
    return codecs.encode(dense_product(W, X, dt, alpha, rows), out_dt)


def gemm_sp24(values: np.ndarray, meta: np.ndarray, K: int, X: np.ndarray, dt: str,
              out_dt: str, alpha: float = 1.0, rows=None) -> np.ndarray:
    """Y = round_out(alpha * decompress(values, meta) . X) as output-type bits."""
    if rows is not None:
        values, meta = values[rows], meta[rows]
    W_hat = sp24.decompress(values, meta, K)
    return gemm_dense(W_hat, X, dt, out_dt, alpha)


def within_bound(Y_bits: np.ndarray, Y_ref_bits: np.ndarray, B: np.ndarray, out_dt: str,
                 rel: float) -> np.ndarray:
    """Elementwise |Y - Y_ref| <= rel * B (equality where B == 0)."""
    y = codecs.decode(Y_bits, out_dt)
    r = codecs.decode(Y_ref_bits, out_dt)
    d = np.abs(y - r)
    ok = d <= rel * B
    return ok & np.isfinite(y)
