"""Indexer scores and per-query top-K selection (CSA2 FULL / REINDEX / REUSE).

Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression",
picx.dev summary, Methodology / Architecture Components / 2. Compressed Sparse
Attention 2: a FULL layer computes its own indexer K and top-K indices, a
REINDEX layer computes fresh top-K indices, a REUSE layer takes the preceding
layer's indices unchanged.

Hierarchical Sparse Indexer (same summary, Methodology / 3): the first FULL
layer's selection builds a candidate pool of at most 2,048 blocks x 8
positions that bounds the search of the REINDEX layers after it.

Readings (the page names the indexer but prints no formula):
  * score I[n] = sum_h w[h] * max(0, q[h] . z[n]) over H_I indexer heads, with
    a per-query weight vector w (the multi-head ReLU scalar score);
  * top-K keeps the K largest scores among the visible entries n < n_visible;
    equal scores go to the lower index; the result is listed in ascending
    index order and padded with -1 when fewer than K entries are visible;
  * a pool block is an aligned run of 8 compressed positions (8b .. 8b+7); the
    pool of a query is the union of the blocks that hold an entry of the FULL
    layer's selection for that query (at most K blocks, 8K positions), and a
    REINDEX layer given that selection ranks only the pool's visible positions
    with its own indexer query and keys, under the same top-K rules.
"""
from __future__ import annotations

import numpy as np


def scores(q_idx: np.ndarray, w_idx: np.ndarray, z: np.ndarray) -> np.ndarray:
    """I[t, n] for one sequence: q_idx [T, H_I, D_I], w_idx [T, H_I], z [N, D_I] -> [T, N] float64."""
    q = np.asarray(q_idx, dtype=np.float64)
    w = np.asarray(w_idx, dtype=np.float64)
    zz = np.asarray(z, dtype=np.float64)
    dots = np.einsum("thd,nd->thn", q, zz)             # per-head dot products
    return np.einsum("th,thn->tn", w, np.maximum(dots, 0.0))


def topk(score_row: np.ndarray, n_visible: int, K: int) -> np.ndarray:
    """Indices of the K best visible entries, ascending, -1 padded (int32 [K])."""
    n_visible = int(n_visible)
    s = np.asarray(score_row[:n_visible], dtype=np.float64)
    order = np.lexsort((np.arange(n_visible), -s))     # primary: score desc; secondary: index asc
    take = np.sort(order[: min(K, n_visible)])
    out = np.full(K, -1, dtype=np.int32)
    out[: take.size] = take
    return out


def kth_score(score_row: np.ndarray, n_visible: int, K: int) -> float:
    """Score of the K-th selected entry (the selection threshold), or -inf if all are taken."""
    s = np.sort(np.asarray(score_row[: int(n_visible)], dtype=np.float64))[::-1]
    if K >= s.size or s.size == 0:
        return -np.inf
    return float(s[K - 1])


POOL_BLOCK = 8   # positions per block of the candidate pool


def candidate_pool(full_idx: np.ndarray, block: int = POOL_BLOCK) -> np.ndarray:
    """Positions of the candidate pool built from one query's FULL-layer selection
    full_idx [K] (-1 padded): every position of every aligned block that holds a selected
    entry, ascending (int64)."""
    sel = np.asarray(full_idx, dtype=np.int64)
    sel = sel[sel >= 0]
    blocks = np.unique(sel // block)
    return (blocks[:, None] * block + np.arange(block)[None, :]).reshape(-1)


def topk_in_pool(score_row: np.ndarray, n_visible: int, K: int, pool: np.ndarray) -> np.ndarray:
    """topk restricted to the pool's visible positions (int32 [K], ascending, -1 padded)."""
    pool = np.asarray(pool, dtype=np.int64)
    cand = pool[pool < int(n_visible)]
    s = np.asarray(score_row, dtype=np.float64)[cand]
    order = np.lexsort((cand, -s))                     # score desc, then position asc
    take = np.sort(cand[order[: min(K, cand.size)]])
    out = np.full(K, -1, dtype=np.int32)
    out[: take.size] = take
    return out


def index_topk(mode: int, q_idx, w_idx, z, n_visible, K: int, prev_idx=None):
    """One sequence's indices for a layer of the given mode (0 FULL, 1 REINDEX, 2 REUSE,
    3 REINDEX over the candidate pool of prev_idx).

    FULL and REINDEX compute the same thing from their own query and keys (the
    difference between them is which main KV the attention reads); REUSE
    returns the preceding layer's indices. The pool mode takes prev_idx as the first FULL
    layer's selection ([T, K]) and searches only each query's candidate pool.
    """
    if mode == 2:
        if prev_idx is None:
            raise ValueError("REUSE needs the preceding layer's indices")
        return np.array(prev_idx, dtype=np.int32, copy=True)
    I = scores(q_idx, w_idx, z)
    T = I.shape[0]
    if mode == 3:
        if prev_idx is None:
            raise ValueError("the pool mode needs the FULL layer's selection")
        return np.stack([topk_in_pool(I[t], n_visible[t], K, candidate_pool(prev_idx[t])) for t in range(T)])
    return np.stack([topk(I[t], n_visible[t], K) for t in range(T)])
