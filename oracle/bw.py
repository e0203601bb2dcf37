"""Block-wise (BW) sparsity in the tiled-GEMM form.

"Accelerating Sparse DNNs Based on Tiled GEMM": Abstract (tile-vector-wise
sparsity is compared with block sparsity, 2.75x), Figure 5 caption (the EW, VW
and BW pruning algorithms). Block sparsity removes whole blocks of weights.

Readings where the pages are silent (each also listed in the design notes):
  * a block is 128 rows of W (one GEMM tile, as in tile-wise sparsity) by 64
    consecutive columns (one K step of the tiled GEMM for 16-bit data); K % 64 == 0;
  * block score = fp32 sum over the block's 64 columns, in ascending column order,
    of the tile-wise column scores s_t[k] (each the fp32 sum over the tile's rows,
    in ascending row order, of |w_ik|);
  * tile t keeps the first B_t blocks of the order (score descending, block index
    ascending), listed in ascending block index;
  * the packed operand is the tile-wise packed operand of the kept columns (the
    kept blocks' columns, L_t = 64 B_t), and the tile schedule is the tile-wise one
    for those L_t.

Layouts (the library's contract, restated):
  offsets[t] = sum_{s<t} B_s (T + 1 entries), counted in blocks;
  indices[offsets[t] + i] = the i-th kept block of tile t (ascending);
  packed: element (t, r, j), j < 64 B_t, at 128 P_t + 8192 (j // 64) + 64 r + j % 64
      with P_t = sum_{s<t} 64 B_s; zero where row 128 t + r >= M.
"""
from __future__ import annotations

import numpy as np

from . import codecs, tw
from . import gemm as products

T = 128
BW = 64


def block_scores(W: np.ndarray, dt: str) -> np.ndarray:
    """bs[t, b] = fp32 sum over j = 0..63, ascending, of s_t[64 b + j]."""
    s = tw.scores(W, dt)
    nt, K = s.shape
    assert K % BW == 0
    s3 = s.reshape(nt, K // BW, BW)
    acc = np.zeros((nt, K // BW), dtype=np.float32)
    for j in range(BW):
        acc = acc + s3[:, :, j]                              # one fp32 add per column, in column order
    return acc


def prune(W: np.ndarray, dt: str, keep_blocks: np.ndarray) -> dict:
    """The BW compressed form of W for per-tile kept block counts `keep_blocks`."""
    M, K = W.shape
    assert K % BW == 0
    nt = (M + T - 1) // T
    KB = K // BW
    keep_blocks = np.asarray(keep_blocks, dtype=np.int64)
    assert keep_blocks.shape == (nt,) and np.all((keep_blocks >= 0) & (keep_blocks <= KB))
    bs = block_scores(W, dt)
    L = BW * keep_blocks
    P = np.concatenate([[0], np.cumsum(L)])
    packed = np.zeros(T * int(P[-1]), dtype=W.dtype)
    blk_all, col_all = [], []
    for t in range(nt):
        blocks = tw.select(bs[t], int(keep_blocks[t]))
        cols = (BW * blocks[:, None] + np.arange(BW)[None, :]).reshape(-1).astype(np.int32)
        blk_all.append(blocks)
        col_all.append(cols)
        g = tw.gathered_tile(W, t, cols)                      # 128 x L_t
        for j0 in range(0, int(L[t]), BW):
            base = T * int(P[t]) + T * j0
            packed[base:base + T * BW] = g[:, j0:j0 + BW].reshape(-1)
    cat = lambda parts: np.concatenate(parts).astype(np.int32) if parts else np.zeros(0, np.int32)
    return {"offsets": tw.offsets_of(keep_blocks), "indices": cat(blk_all), "col_indices": cat(col_all),
            "schedule_table": tw.schedule_table(L), "packed": packed, "block_scores": bs}


def unpack_tile(form: dict, keep_blocks: np.ndarray, t: int) -> np.ndarray:
    """The 128 x 64 B_t kept block of tile t, rebuilt from the packed operand."""
    L = BW * np.asarray(keep_blocks, dtype=np.int64)
    P = np.concatenate([[0], np.cumsum(L)])
    blk = np.zeros((T, int(L[t])), dtype=form["packed"].dtype)
    for j0 in range(0, int(L[t]), BW):
        base = T * int(P[t]) + T * j0
        blk[:, j0:j0 + BW] = form["packed"][base:base + T * BW].reshape(T, BW)
    return blk


def masked_dense(W: np.ndarray, form: dict, keep_blocks: np.ndarray) -> np.ndarray:
    """W with every block that is not kept set to zero (rows past M dropped)."""
    M, K = W.shape
    out = np.zeros_like(W)
    off = form["offsets"]
    for t in range(len(keep_blocks)):
        r0, r1 = t * T, min(M, (t + 1) * T)
        for b in form["indices"][off[t]:off[t + 1]]:
            out[r0:r1, BW * b:BW * (b + 1)] = W[r0:r1, BW * b:BW * (b + 1)]
    return out


def gemm(form: dict, keep_blocks: np.ndarray, X: np.ndarray, dt: str, out_dt: str, M: int, alpha: float = 1.0,
         tiles=None) -> tuple[np.ndarray, np.ndarray]:
    """Y (M x N output bits) and its error bound B: Y[tile t] = round(alpha * W_t . X[kept rows])."""
    N = X.shape[1]
    nt = len(keep_blocks)
    Xd = codecs.decode(X, dt)
    Yf = np.zeros((nt * T, N))
    B = np.zeros((nt * T, N))
    off = form["offsets"]
    for t in (range(nt) if tiles is None else tiles):
        cols = form["col_indices"][BW * off[t]:BW * off[t + 1]]
        Wt = codecs.decode(unpack_tile(form, keep_blocks, t), dt)
        Yf[t * T:(t + 1) * T] = alpha * (Wt @ Xd[cols])
        B[t * T:(t + 1) * T] = products.bound_decoded(Wt, Xd[cols], alpha)
    return codecs.encode(Yf[:M], out_dt), B[:M]
