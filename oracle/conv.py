"""3x3 convolution (stride 1, zero padding 1) with a 2:4-sparse or dense filter.

"SparseRT: Accelerating Unstructured Sparsity on GPUs for Deep Learning
Inference", Abstract: sparse 3x3 convolutions (ResNet-50 use cases) beside the
1x1 / fully connected ones. "Accelerating Sparse Deep Neural Networks", Abstract:
2:4 sparsity applies to the convolution's weight the same way as to a GEMM's.

Readings where the pages are silent (each also listed in the design notes):
  * activations X are NHWC (batch, H, W, C_in); the filter is (C_out, 3, 3, C_in),
    flattened to a C_out x 9 C_in matrix whose column (r 3 + s) C_in + c holds
    tap (r, s) of input channel c;
  * 2:4 applies along that flattened K (groups of four consecutive input channels
    of one tap), i.e. it is the 2:4 compression of the flattened filter;
  * Y[co, (n H + h) W + w] = alpha * sum_{r, s, c} W[co, r, s, c] X[n, h + r - 1, w + s - 1, c]
    (zero outside the image): the output is C_out x (N H W), channel-major;
  * numerics as the GEMM: fp64 sum, one rounding to the output type;
  * tile-wise filter ("Accelerating Sparse DNNs Based on Tiled GEMM", Abstract:
    whole K-rows of the GEMM pruned per output tile, the skip made where operands
    are fetched): a 128-channel output tile keeps whole K-row groups of one tap and
    64 input channels (the unit in which the implicit GEMM fetches activations);
    group g is columns 64 g .. 64 g + 63 of the flattened filter, scored by the fp32
    sum of its columns' tile-wise scores -- the block-wise selection of bw.prune with
    64-column blocks -- and the convolution uses the filter masked to those groups.
"""
from __future__ import annotations

import numpy as np

from . import bw, codecs, gemm, sp24


def im2col(X: np.ndarray) -> np.ndarray:
    """The (9 C_in) x (N H W) matrix of the definition: row (r 3 + s) C_in + c,
    column (n H + h) W + w holds X[n, h + r - 1, w + s - 1, c] (0 outside)."""
    Nb, H, W, Cin = X.shape
    Xp = np.zeros((Nb, H + 2, W + 2, Cin), dtype=X.dtype)
    Xp[:, 1:H + 1, 1:W + 1, :] = X
    cols = np.zeros((9 * Cin, Nb * H * W), dtype=X.dtype)
    for r in range(3):
        for s in range(3):
            tap = Xp[:, r:r + H, s:s + W, :]                       # X[n, h + r - 1, w + s - 1, c]
            cols[(3 * r + s) * Cin:(3 * r + s + 1) * Cin] = tap.reshape(-1, Cin).T
    return cols


def conv3x3(Wf: np.ndarray, X: np.ndarray, dt: str, out_dt: str, alpha: float = 1.0,
            sparse: bool = True) -> tuple[np.ndarray, np.ndarray]:
    """Y bits (C_out x N H W) and the elementwise bound, for a filter Wf of shape
    (C_out, 9 C_in) bits (2:4-pruned first when `sparse`)."""
    if sparse:
        v, m = sp24.compress(Wf, dt)
        Wf = sp24.decompress(v, m, Wf.shape[1])
    cols = im2col(X)
    Y = gemm.dense_product(Wf, cols, dt, alpha)
    B = gemm.bound(Wf, cols, dt, alpha)
    return codecs.encode(Y, out_dt), B


def conv3x3_tw(Wf: np.ndarray, X: np.ndarray, dt: str, out_dt: str, keep_groups, alpha: float = 1.0):
    """Y bits and bound for the tile-wise filter: per 128-channel tile t the first
    keep_groups[t] (tap, 64-channel) groups by score (ties to the lower group), the
    rest of the filter zero. Returns (Y, B, form) with form = bw.prune's output."""
    keep = np.asarray(keep_groups, dtype=np.int64)
    form = bw.prune(Wf, dt, keep)
    masked = bw.masked_dense(Wf, form, keep)
    Y, B = conv3x3(masked, X, dt, out_dt, alpha, sparse=False)
    return Y, B, form


def conv3x3_direct(Wf: np.ndarray, X: np.ndarray, dt: str) -> np.ndarray:
    """The convolution sum written out with loops over taps and pixels (fp64 values,
    dense filter): the independent form the im2col path is pinned against."""
    Nb, H, W, Cin = X.shape
    Cout = Wf.shape[0]
    w = codecs.decode(Wf, dt).reshape(Cout, 3, 3, Cin)
    x = codecs.decode(X, dt)
    Y = np.zeros((Cout, Nb, H, W))
    for n in range(Nb):
        for h in range(H):
            for ww in range(W):
                for r in range(3):
                    for s in range(3):
                        hh, wx = h + r - 1, ww + s - 1
                        if 0 <= hh < H and 0 <= wx < W:
                            Y[:, n, h, ww] += w[:, r, s, :] @ x[n, hh, wx, :]
    return Y.reshape(Cout, Nb * H * W)
