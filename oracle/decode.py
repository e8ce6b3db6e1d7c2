"""One CSA2 layer group end to end on the CPU, following the layer modes.

Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression",
picx.dev summary, Methodology / 2. Compressed Sparse Attention 2:
  FULL     own main KV (FP4-encoded here), own indexer keys, own top-K;
  REINDEX  the preceding layer's main KV, fresh top-K from its own indexer;
  REUSE    the preceding layer's main KV and top-K indices.
Each layer then attends over its selected entries (global branch) and over the
last n_win raw tokens (SWA branch) and combines the two by LSE.
"""
from __future__ import annotations

import numpy as np

from . import attention, fp4, indexer


def layer_outputs(mode, q, kv_rows, idx, swa_rows, win_start, win_len, d_v, tau):
    """All queries of one sequence: q [T, H, 576] -> dict with O_g, LSE_g, O, LSE ([T, H, ...])."""
    T, H, _ = q.shape
    Og = np.zeros((T, H, d_v)); Lg = np.zeros((T, H))
    O = np.zeros((T, H, d_v)); L = np.zeros((T, H))
    for t in range(T):
        og, lg = attention.sparse_global(q[t], kv_rows, idx[t], d_v, tau)
        os_, ls = attention.swa_branch(q[t], swa_rows, int(win_start[t]), int(win_len[t]), d_v, tau)
        o, l = attention.merge(og, lg, os_, ls)
        Og[t], Lg[t], O[t], L[t] = og, lg, o, l
    return dict(O_g=Og, LSE_g=Lg, O=O, LSE=L)


def run_group_sequence(layers, b, n_visible, win_start, win_len, K, d_v, tau, bf16_to_f64):
    """Run every layer of a group for batch element b.

    layers: sequence of objects with fields mode, X, z, q_idx, w_idx, q, swa
    (bf16 given as bit patterns, converted with bf16_to_f64). Returns a list of
    per-layer dicts with idx, codes, scales and the attention outputs.
    """
    out = []
    kv_codes = kv_scales = kv_rows = None
    prev_idx = None
    for L in layers:
        T = L.q.shape[1]
        nv = n_visible[b * T:(b + 1) * T]
        ws = win_start[b * T:(b + 1) * T]
        wl = win_len[b * T:(b + 1) * T]
        if L.mode == 0:
            kv_codes, kv_scales = fp4.encode(L.X[b])
            kv_rows = fp4.decode(kv_codes, kv_scales)
        if L.mode in (0, 1):
            idx = indexer.index_topk(L.mode, bf16_to_f64(L.q_idx[b]), L.w_idx[b], bf16_to_f64(L.z[b]), nv, K)
        else:
            idx = indexer.index_topk(2, None, None, None, nv, K, prev_idx=prev_idx)
        res = layer_outputs(L.mode, bf16_to_f64(L.q[b]), kv_rows, idx, bf16_to_f64(L.swa[b]), ws, wl, d_v, tau)
        res.update(idx=idx, codes=kv_codes, scales=kv_scales)
        out.append(res)
        prev_idx = idx
    return out
