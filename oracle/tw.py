"""Tile-wise (TW) and tile-vector-wise (TVW) sparsity.

"Accelerating Sparse DNNs Based on Tiled GEMM": TL;DR and Abstract (a pattern
that is regular inside each GEMM tile but irregular across tiles; TW applied at
the global-memory level, 2:4 applied inside the sparse tensor core; the two
combined as TVW; batching of tiles for load balance), Figure 3 caption (the TW
pattern follows the tiled GEMM).

Readings where the pages are silent (each also listed in the design notes):
  * a tile is T = 128 consecutive rows of W (output features); tile t keeps a
    set of L_t column indices k of W, i.e. rows of X, for all of its rows;
  * score s_t[k] = sum over the tile's rows i, in ascending i, of |w_ik| in fp32;
  * the kept set is the first L_t of the order (score descending, k ascending),
    listed in ascending k;
  * TVW applies the 2:4 rule along the compacted K of each packed tile
    (groups of four consecutive kept columns), so L_t % 4 == 0;
  * schedule ("load-balancing through batching"): tiles in order of L_t
    descending, ties by t ascending; equal L_t form one batch. The table form
    lists (t, L_t, P_t, Q_t = P_t / 64) per tile in that order.

Layouts (the library's contract, restated):
  R_t = round_up(L_t, 64), P_t = sum_{s<t} R_s.
  offsets[t] = sum_{s<t} L_s (T + 1 entries); indices[offsets[t] + j] = j-th kept k.
  TW packed (dense): element (t, r, j), j < R_t, at 128 P_t + 8192 (j // 64)
      + 64 r + j % 64; zero where j >= L_t or row 128 t + r >= M.
  TVW values: (t, r, c), c < R_t / 2, at 64 P_t + 4096 (c // 32) + 32 r + c % 32.
  TVW meta (canonical): byte b < R_t / 8 of tile row r at 16 P_t + r R_t / 8 + b.
  TVW meta_hw: tile t owns R_t / 64 blocks of 2048 bytes starting at block
      Q_t = P_t / 64: the 16-bit operand layout of sp24.meta_hw_from_canonical
      applied to the tile's canonical metadata (128 rows, K = R_t).
"""
from __future__ import annotations

import numpy as np

from . import codecs, sp24
from . import gemm as products

T = 128
U = 64


def scores(W: np.ndarray, dt: str) -> np.ndarray:
    """s[t, k] = fp32 sum over the tile's rows, ascending, of |w_ik|."""
    M, K = W.shape
    nt = (M + T - 1) // T
    a = np.abs(codecs.decode(W, dt)).astype(np.float32)   # |w| is exact in fp32
    s = np.zeros((nt, K), dtype=np.float32)
    for t in range(nt):
        acc = np.zeros(K, dtype=np.float32)
        for i in range(t * T, min(M, (t + 1) * T)):
            acc = acc + a[i]                                 # one fp32 add per row, in row order
        s[t] = acc
    return s


def select(s_t: np.ndarray, L: int) -> np.ndarray:
    """Indices of the first L of (score descending, k ascending), sorted ascending."""
    K = s_t.shape[0]
    k = np.arange(K)
    order = np.lexsort((k, -s_t.astype(np.float64)))
    return np.sort(order[:L]).astype(np.int32)


def offsets_of(keep: np.ndarray) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(keep)]).astype(np.int32)


def schedule(keep: np.ndarray) -> np.ndarray:
    """Tiles ordered by kept count descending, ties by tile index ascending."""
    t = np.arange(len(keep))
    return np.lexsort((t, -keep.astype(np.int64))).astype(np.int32)


def padded(L: np.ndarray) -> np.ndarray:
    return (L + U - 1) // U * U


def schedule_table(keep: np.ndarray) -> np.ndarray:
    """(t, L_t, P_t, Q_t) for the tiles in schedule order, flattened (4 per tile)."""
    keep = np.asarray(keep, dtype=np.int64)
    R = padded(keep)
    P = np.concatenate([[0], np.cumsum(R)])[:-1]
    Q = P // 64
    order = schedule(keep)
    return np.stack([order, keep[order], P[order], Q[order]], axis=1).reshape(-1).astype(np.int32)


def gathered_tile(W: np.ndarray, t: int, idx: np.ndarray) -> np.ndarray:
    """The 128 x L_t block W[tile rows][idx] (rows past M are zero)."""
    M, K = W.shape
    blk = np.zeros((T, len(idx)), dtype=W.dtype)
    r1 = min(M, (t + 1) * T)
    blk[: r1 - t * T] = W[t * T:r1][:, idx]
    return blk


def prune(W: np.ndarray, dt: str, keep: np.ndarray, tvw: bool) -> dict:
    """The TW (or TVW) compressed form of W for per-tile kept counts `keep`."""
    M, K = W.shape
    nt = (M + T - 1) // T
    keep = np.asarray(keep, dtype=np.int64)
    assert keep.shape == (nt,) and np.all((keep >= 0) & (keep <= K))
    if tvw:
        assert np.all(keep % 4 == 0)
    s = scores(W, dt)
    R = padded(keep)
    P = np.concatenate([[0], np.cumsum(R)])
    idx_all = []
    packed = np.zeros(T * int(P[-1]) // (2 if tvw else 1), dtype=W.dtype)
    meta = np.full(16 * int(P[-1]), 0x44, dtype=np.uint8) if tvw else None
    meta_hw = np.zeros(32 * int(P[-1]), dtype=np.uint8) if tvw else None
    for t in range(nt):
        L, Rt, Pt = int(keep[t]), int(R[t]), int(P[t])
        idx = select(s[t], L)
        idx_all.append(idx)
        blk = np.zeros((T, Rt), dtype=W.dtype)
        blk[:, :L] = gathered_tile(W, t, idx)
        if not tvw:
            for j0 in range(0, Rt, U):
                base = T * Pt + T * j0
                packed[base:base + T * U] = blk[:, j0:j0 + U].reshape(-1)
        else:
            vals, m = sp24.compress(blk[:, :L], dt) if L > 0 else (np.zeros((T, 0), W.dtype), np.zeros((T, 0), np.uint8))
            v = np.zeros((T, Rt // 2), dtype=W.dtype)
            v[:, :L // 2] = vals[:, :L // 2]
            for c0 in range(0, Rt // 2, U // 2):
                base = T * Pt // 2 + T * c0
                packed[base:base + T * (U // 2)] = v[:, c0:c0 + U // 2].reshape(-1)
            mc = np.full((T, Rt // 8), 0x44, dtype=np.uint8)
            nbytes = min(m.shape[1], Rt // 8)
            mc[:, :nbytes] = m[:, :nbytes]
            meta[16 * Pt:16 * Pt + T * (Rt // 8)] = mc.reshape(-1)
            if Rt:
                hw = sp24.meta_hw_from_canonical(mc, T, Rt, dt)
                meta_hw[32 * Pt:32 * Pt + hw.size] = hw
    indices = np.concatenate(idx_all).astype(np.int32) if idx_all else np.zeros(0, np.int32)
    return {"offsets": offsets_of(keep), "indices": indices, "schedule": schedule(keep),
            "schedule_table": schedule_table(keep),
            "packed": packed, "meta": meta, "meta_hw": meta_hw, "scores": s}


def unpack_tile(form: dict, keep: np.ndarray, t: int, tvw: bool, dt: str) -> np.ndarray:
    """The 128 x L_t kept block of tile t, rebuilt from the packed form."""
    keep = np.asarray(keep, dtype=np.int64)
    R = padded(keep)
    P = np.concatenate([[0], np.cumsum(R)])
    L, Rt, Pt = int(keep[t]), int(R[t]), int(P[t])
    if not tvw:
        blk = np.zeros((T, Rt), dtype=form["packed"].dtype)
        for j0 in range(0, Rt, U):
            base = T * Pt + T * j0
            blk[:, j0:j0 + U] = form["packed"][base:base + T * U].reshape(T, U)
        return blk[:, :L]
    v = np.zeros((T, Rt // 2), dtype=form["packed"].dtype)
    for c0 in range(0, Rt // 2, U // 2):
        base = T * Pt // 2 + T * c0
        v[:, c0:c0 + U // 2] = form["packed"][base:base + T * (U // 2)].reshape(T, U // 2)
    mc = form["meta"][16 * Pt:16 * Pt + T * (Rt // 8)].reshape(T, Rt // 8)
    return sp24.decompress(v[:, :L // 2], mc, L)


def gemm(form: dict, keep: np.ndarray, X: np.ndarray, dt: str, out_dt: str, M: int,
         tvw: bool, alpha: float = 1.0, tiles=None) -> tuple[np.ndarray, np.ndarray]:
    """Y (M x N output bits) and its error bound B for the TW / TVW form.

    Y[tile t rows] = round_out(alpha * W_t . X[idx_t, :]); an empty tile gives +0.
    Only the tiles in `tiles` are computed when given (other rows are zero).
    """
    N = X.shape[1]
    keep = np.asarray(keep, dtype=np.int64)
    nt = len(keep)
    off = form["offsets"]
    Xd = codecs.decode(X, dt)
    Yf = np.zeros((nt * T, N))
    B = np.zeros((nt * T, N))
    for t in (range(nt) if tiles is None else tiles):
        idx = form["indices"][off[t]:off[t + 1]]
        Wt = codecs.decode(unpack_tile(form, keep, t, tvw, dt), dt)
        Xt = Xd[idx]
        Yf[t * T:(t + 1) * T] = alpha * (Wt @ Xt)
        B[t * T:(t + 1) * T] = products.bound_decoded(Wt, Xt, alpha)
    return codecs.encode(Yf[:M], out_dt), B[:M]
