"""Sparse MQA over selected entries, the sliding-window branch, and their LSE merge.

Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression":
  * cyber-feed.org blog repost, paragraph on the DeepSeek-V4 architecture: a
    sparse attention branch that covers the whole context is combined with a
    sliding-window attention (SWA) branch over the local window;
  * picx.dev summary, Introduction and Theoretical Foundation (global branch
    plus local SWA) and Methodology / 2. CSA2 (the global KV and its top-K);
  * wesearch.press card: head-count reduction (one KV shared by all query heads).

Readings where the pages are silent:
  * one latent entry (576 = 512 latent + 64 rope) is both key and value; the
    value is its first d_v channels (512), the rope channels are key-only;
  * scores are tau * q_h . k_j with tau = 1/sqrt(576); softmax per head;
  * the two branches are combined as one softmax over the union of their key
    sets, i.e. by log-sum-exp weighting of the two normalised outputs;
  * outputs are float64 here (float32 on the device); an empty key set gives
    O = 0 and LSE = -inf.
"""
from __future__ import annotations

import numpy as np


def attend(q: np.ndarray, keys: np.ndarray, d_v: int, tau: float):
    """Softmax attention of q [H, D] over keys [n, D] (values = keys[:, :d_v]).

    Returns (O [H, d_v], LSE [H]) in float64 with natural-log LSE.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(keys, dtype=np.float64)
    H = q.shape[0]
    if k.shape[0] == 0:
        return np.zeros((H, d_v)), np.full(H, -np.inf)
    s = tau * (q @ k.T)                                  # [H, n]
    m = np.max(s, axis=1, keepdims=True)
    p = np.exp(s - m)
    l = np.sum(p, axis=1, keepdims=True)
    O = (p @ k[:, :d_v]) / l
    lse = (m + np.log(l))[:, 0]
    return O, lse


def merge(O_a, lse_a, O_b, lse_b):
    """Combine two normalised partial attentions over disjoint key sets.

    The result equals one softmax over the union: weights exp(LSE_x - LSE).
    """
    lse_a = np.asarray(lse_a, dtype=np.float64)
    lse_b = np.asarray(lse_b, dtype=np.float64)
    lse = np.logaddexp(lse_a, lse_b)
    with np.errstate(invalid="ignore"):
        wa = np.where(np.isneginf(lse_a), 0.0, np.exp(lse_a - lse))
        wb = np.where(np.isneginf(lse_b), 0.0, np.exp(lse_b - lse))
    O = wa[:, None] * np.asarray(O_a, dtype=np.float64) + wb[:, None] * np.asarray(O_b, dtype=np.float64)
    empty = np.isneginf(lse)
    O[empty] = 0.0
    return O, lse


def sparse_global(q, kv_dequant_rows: np.ndarray, idx: np.ndarray, d_v: int, tau: float):
    """Global branch for one query: attend over the rows named by idx (-1 entries skipped)."""
    sel = np.asarray(idx)
    sel = sel[sel >= 0]
    return attend(q, kv_dequant_rows[sel], d_v, tau)


def swa_branch(q, swa_rows: np.ndarray, start: int, length: int, d_v: int, tau: float):
    """Sliding-window branch for one query over raw rows [start, start+length)."""
    return attend(q, swa_rows[start:start + length], d_v, tau)
