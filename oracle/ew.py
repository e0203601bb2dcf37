"""Element-wise (EW, unstructured) sparsity and the sparse x dense product.

"SparseRT: Accelerating Unstructured Sparsity on GPUs for Deep Learning
Inference", Abstract: weights pruned individually (unstructured sparsity) at
90 % and 95 % sparsity, 1x1 convolutions and fully connected layers computed as a
sparse weight matrix times a dense activation matrix. "Accelerating Sparse DNNs
Based on Tiled GEMM", Abstract and Figure 5 caption: EW pruning is the
unstructured comparison point of tile-vector-wise sparsity (22.18x).

Readings where the pages are silent (each also listed in the design notes):
  * magnitude pruning with the same kept count k in every row of W (so rows are
    balanced): row i keeps the first k of (|w_ik| descending, k ascending),
    |w| ordered by the stored bits with the sign cleared (as for 2:4), listed in
    ascending column order; k = round(density * K) is the caller's choice;
  * the compressed form is CSR: row_ptr[i] = i k, col_idx and the kept values'
    stored bits in row order;
  * the product Y = W_ew . X accumulates in fp32 on the device; the oracle
    computes it in fp64 (one rounding to the output type), checked within the
    elementwise bound like the other GEMMs.
"""
from __future__ import annotations

import numpy as np

from . import codecs
from . import gemm as products

_MAG = {"f16": 0x7FFF, "bf16": 0x7FFF, "e4m3": 0x7F}


def select_row(w_row: np.ndarray, k: int, dt: str) -> np.ndarray:
    """Column indices of the first k of (magnitude bits descending, index ascending), sorted."""
    mag = (w_row.astype(np.int64) & _MAG[dt])
    order = np.lexsort((np.arange(w_row.shape[0]), -mag))
    return np.sort(order[:k]).astype(np.int32)


def prune(W: np.ndarray, dt: str, k: int) -> dict:
    """CSR form of W keeping k entries per row."""
    M, K = W.shape
    assert 0 <= k <= K
    col = np.zeros((M, k), dtype=np.int32)
    for i in range(M):
        col[i] = select_row(W[i], k, dt)
    vals = np.take_along_axis(W, col.astype(np.int64), axis=1)
    return {"row_ptr": (np.arange(M + 1) * k).astype(np.int32), "col_idx": col.reshape(-1),
            "vals": vals.reshape(-1), "k": k}


def decompress(form: dict, M: int, K: int) -> np.ndarray:
    """Dense bits of the pruned W (zeros elsewhere)."""
    k = form["k"]
    W = np.zeros((M, K), dtype=form["vals"].dtype)
    rows = np.repeat(np.arange(M), k)
    W[rows, form["col_idx"]] = form["vals"]
    return W


def spmm(form: dict, M: int, K: int, X: np.ndarray, dt: str, out_dt: str, alpha: float = 1.0,
         rows=None) -> tuple[np.ndarray, np.ndarray]:
    """Y bits = round(alpha * W_ew . X) and the bound B = |alpha| sum |w x| (fp64),
    optionally on a subset of rows."""
    k = form["k"]
    r = np.arange(M) if rows is None else np.asarray(rows)
    Xd = codecs.decode(X, dt)
    cols_all = form["col_idx"].reshape(M, k)
    vals_all = form["vals"].reshape(M, k)
    Y = np.zeros((len(r), X.shape[1]))
    B = np.zeros((len(r), X.shape[1]))
    for j, i in enumerate(r):                     # one row at a time: sum_k w_ik x_k
        w = codecs.decode(vals_all[i], dt)
        xk = Xd[cols_all[i]]
        Y[j] = alpha * (w @ xk)
        B[j] = products.bound_decoded(w, xk, alpha)
    return codecs.encode(Y, out_dt), B
