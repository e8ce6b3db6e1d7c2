"""Pins of the oracle's indexer scores and top-K selection (no GPU).

Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", picx.dev summary,
Methodology / 2. CSA2 (FULL/REINDEX compute top-K indices, REUSE takes the preceding ones).
"""
import numpy as np

from oracle import indexer


def test_closed_form_two_heads():
    """w = [2, 3], q0 = e0, q1 = -e1, z_n = (n, n-3, 0, ...): I(n) = 2*max(0, n) + 3*max(0, 3-n).

    Catches a ReLU applied after the head sum, a dropped weight or a transposed operand."""
    N, D = 8, 64
    z = np.zeros((N, D))
    z[:, 0] = np.arange(N) - 2            # n - 2, so some dots are negative
    z[:, 1] = np.arange(N) - 3
    q = np.zeros((1, 2, D)); q[0, 0, 0] = 1.0; q[0, 1, 1] = -1.0
    w = np.array([[2.0, 3.0]])
    got = indexer.scores(q, w, z)[0]
    n = np.arange(N)
    want = 2 * np.maximum(0, n - 2) + 3 * np.maximum(0, 3 - n)
    assert np.array_equal(got, want)


def _select_by_loop(s, n_visible, K):
    chosen = []
    alive = list(range(n_visible))
    for _ in range(min(K, n_visible)):
        best = alive[0]
        for i in alive[1:]:
            if s[i] > s[best]:
                best = i          # strict: equal scores keep the lower index
        chosen.append(best)
        alive.remove(best)
    out = sorted(chosen) + [-1] * (K - len(chosen))
    return out


def test_topk_matches_brute_force_with_ties():
    rng = np.random.default_rng(3)
    for trial in range(300):
        N = int(rng.integers(1, 40))
        s = rng.integers(0, 6, size=N).astype(float)     # many ties
        nv = int(rng.integers(0, N + 1))
        K = int(rng.integers(1, 45))
        assert list(indexer.topk(s, nv, K)) == _select_by_loop(s, nv, K)


def test_k_at_least_n_visible_selects_everything():
    s = np.random.default_rng(4).standard_normal(100)
    out = indexer.topk(s, 73, 128)
    assert list(out[:73]) == list(range(73)) and np.all(out[73:] == -1)


def test_all_equal_scores_take_lowest_indices():
    out = indexer.topk(np.zeros(50), 50, 7)
    assert list(out) == list(range(7))


def test_invisible_entries_never_selected():
    s = np.arange(20, dtype=float)        # the best entries are the last ones
    out = indexer.topk(s, 10, 4)
    assert list(out) == [6, 7, 8, 9]


def test_reuse_returns_previous_indices():
    prev = np.array([[3, 5, 9, -1]], dtype=np.int32)
    out = indexer.index_topk(2, None, None, None, [4], 4, prev_idx=prev)
    assert np.array_equal(out, prev) and out is not prev


def test_kth_score():
    s = np.array([5.0, 1.0, 3.0, 4.0])
    assert indexer.kth_score(s, 4, 2) == 4.0
    assert indexer.kth_score(s, 4, 4) == -np.inf
