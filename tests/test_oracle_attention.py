"""Pins of the oracle's sparse attention, SWA branch and LSE merge (no GPU).

Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression": the blog repost
(sparse attention over the whole context combined with a sliding-window branch) and the
picx.dev summary, Methodology / 2. CSA2.
"""
import math

import numpy as np
import pytest

from oracle import attention, fp4, indexer


def _brute(q, keys, d_v, tau):
    """Plain loops with math.exp: an independent statement of softmax attention."""
    H, n = len(q), len(keys)
    O = [[0.0] * d_v for _ in range(H)]
    L = []
    for h in range(H):
        s = [tau * sum(q[h][c] * keys[j][c] for c in range(len(q[h]))) for j in range(n)]
        den = sum(math.exp(x) for x in s)
        for j in range(n):
            p = math.exp(s[j]) / den
            for c in range(d_v):
                O[h][c] += p * keys[j][c]
        L.append(math.log(den))
    return np.array(O), np.array(L)


def test_matches_brute_force_small():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((3, 10))
    keys = rng.standard_normal((7, 10))
    O, L = attention.attend(q, keys, 8, 0.3)
    Ob, Lb = _brute(q.tolist(), keys.tolist(), 8, 0.3)
    assert np.allclose(O, Ob, atol=1e-13) and np.allclose(L, Lb, atol=1e-13)


def test_single_key_and_two_identical_keys():
    q = np.array([[1.0, 2.0, -1.0]])
    k = np.array([[0.5, -1.0, 2.0]])
    O, L = attention.attend(q, k, 2, 1.0)
    assert np.allclose(O, k[:, :2]) and np.isclose(L[0], -3.5)
    O2, L2 = attention.attend(q, np.vstack([k, k]), 2, 1.0)
    assert np.allclose(O2, k[:, :2]) and np.isclose(L2[0], -3.5 + math.log(2))


def test_empty_set():
    O, L = attention.attend(np.ones((2, 4)), np.zeros((0, 4)), 3, 1.0)
    assert np.all(O == 0) and np.all(np.isneginf(L))


def test_merge_equals_one_softmax_over_union():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((4, 16))
    a = rng.standard_normal((9, 16)) * 2
    b = rng.standard_normal((5, 16)) * 2
    Oa, La = attention.attend(q, a, 12, 0.25)
    Ob, Lb = attention.attend(q, b, 12, 0.25)
    O, L = attention.merge(Oa, La, Ob, Lb)
    Ou, Lu = attention.attend(q, np.vstack([a, b]), 12, 0.25)
    assert np.allclose(O, Ou, atol=1e-12) and np.allclose(L, Lu, atol=1e-12)
    # merging with an empty branch is the identity
    Oe, Le = attention.merge(Oa, La, np.zeros_like(Oa), np.full(4, -np.inf))
    assert np.allclose(Oe, Oa) and np.allclose(Le, La)


def test_dominant_key_and_permutation_invariance():
    q = np.array([[10.0, 0.0]])
    keys = np.array([[10.0, 1.0], [0.0, 5.0], [-10.0, 3.0]])
    O, _ = attention.attend(q, keys, 2, 1.0)
    assert np.allclose(O[0], keys[0], atol=1e-30)
    perm = [2, 0, 1]
    O2, L2 = attention.attend(q, keys[perm], 2, 1.0)
    assert np.allclose(O, O2)


def test_full_with_k_at_least_n_equals_dense():
    """With K >= #entries the global branch covers every entry: it equals dense attention."""
    rng = np.random.default_rng(7)
    N = 40
    X = rng.standard_normal((N, 576)).astype(np.float32)
    rows = fp4.decode(*fp4.encode(X))
    qi = rng.standard_normal((1, 2, 64)); wi = np.abs(rng.standard_normal((1, 2))); z = rng.standard_normal((N, 64))
    idx = indexer.index_topk(0, qi, wi, z, [N], 64)[0]
    q = rng.standard_normal((4, 576))
    O, L = attention.sparse_global(q, rows, idx, 512, 1 / 24)
    Od, Ld = attention.attend(q, rows, 512, 1 / 24)
    assert np.allclose(O, Od, atol=1e-12) and np.allclose(L, Ld, atol=1e-12)


def test_padding_entries_are_skipped():
    rng = np.random.default_rng(8)
    rows = rng.standard_normal((10, 8))
    q = rng.standard_normal((2, 8))
    O, L = attention.sparse_global(q, rows, np.array([1, 4, -1, -1]), 6, 0.5)
    O2, L2 = attention.attend(q, rows[[1, 4]], 6, 0.5)
    assert np.allclose(O, O2) and np.allclose(L, L2)


@pytest.mark.parametrize("n_win", [1, 3, 5])
def test_swa_branch_attends_the_last_n_win_tokens(n_win):
    """The window of a query at position p is tokens max(0, p+1-n_win) .. p of the raw store
    (the sliding window of the blog repost, reading R9). Brute force over that token list, at
    positions whose window starts anywhere in the store, the last one ending at its last row."""
    rng = np.random.default_rng(40 + n_win)
    n_tok, D, d_v, tau = 17, 6, 4, 0.4
    store = rng.standard_normal((n_tok, D))
    q = rng.standard_normal((2, D))
    for p in sorted({0, 1, n_win - 1, n_win, n_win + 3, 9, n_tok - 1}):
        if p < 0:
            continue
        window = [store[j].tolist() for j in range(n_tok) if p - n_win < j <= p]
        length = len(window)
        O, L = attention.swa_branch(q, store, p + 1 - length, length, d_v, tau)
        Ob, Lb = _brute(q.tolist(), window, d_v, tau)
        assert np.allclose(O, Ob, atol=1e-13) and np.allclose(L, Lb, atol=1e-13), f"window of token {p}"
