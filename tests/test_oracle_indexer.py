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


# ---- Hierarchical Sparse Indexer (picx.dev summary, Methodology / 3): the first FULL
# layer's selection builds a candidate pool of aligned 8-position blocks that bounds the
# search of the REINDEX layers after it.

def test_candidate_pool_of_a_known_selection():
    """Entries 3, 5 (block 0), 17 (block 2), 100 (block 12) and padding: three blocks."""
    pool = indexer.candidate_pool(np.array([3, 5, 17, 100, -1, -1]))
    want = np.concatenate([np.arange(0, 8), np.arange(16, 24), np.arange(96, 104)])
    assert np.array_equal(pool, want)
    assert indexer.candidate_pool(np.full(4, -1)).size == 0


def test_pool_covering_every_entry_gives_the_full_top_k():
    """When the FULL selection touches every block, the pool is every position and the
    REINDEX result equals the unrestricted top-K (same rules, same ties)."""
    rng = np.random.default_rng(3)
    N, K = 96, 40
    s = np.round(rng.standard_normal(N), 1)            # coarse values: many ties
    full_sel = np.arange(0, N, 8) + rng.integers(0, 8, size=N // 8)
    full_idx = np.full(K, -1)
    full_idx[: full_sel.size] = np.sort(full_sel)
    pool = indexer.candidate_pool(full_idx)
    assert np.array_equal(pool, np.arange(N))
    for nv in (N, 61, 7):
        assert np.array_equal(indexer.topk_in_pool(s, nv, K, pool), indexer.topk(s, nv, K))


def test_pool_top_k_matches_brute_force_and_stays_in_the_pool():
    """Brute force: walk the pool's visible positions, keep the best with a strict
    comparison (ties to the lower position), K times."""
    rng = np.random.default_rng(4)
    N, K = 200, 12
    for trial in range(20):
        s = np.round(rng.standard_normal(N), 1)
        full_idx = np.sort(rng.choice(N, size=9, replace=False))
        pool = indexer.candidate_pool(full_idx)
        nv = int(rng.integers(1, N + 1))
        got = indexer.topk_in_pool(s, nv, K, pool)
        alive = [int(p) for p in pool if p < nv]
        chosen = []
        for _ in range(min(K, len(alive))):
            best = alive[0]
            for i in alive[1:]:
                if s[i] > s[best]:
                    best = i
            chosen.append(best)
            alive.remove(best)
        want = sorted(chosen) + [-1] * (K - len(chosen))
        assert got.tolist() == want, trial
        sel = got[got >= 0]
        assert np.all(np.isin(sel, pool)) and np.all(sel < nv)


def test_pool_size_bound_and_k_covering_the_pool():
    """At most 8 positions per selected entry; with K at least the pool's visible size the
    whole visible pool is selected."""
    rng = np.random.default_rng(5)
    full_idx = np.sort(rng.choice(10_000, size=2048, replace=False))
    pool = indexer.candidate_pool(full_idx)
    assert pool.size <= 8 * 2048 and np.all(np.diff(pool) > 0)
    s = rng.standard_normal(10_000)
    nv = 9_000
    vis = pool[pool < nv]
    got = indexer.topk_in_pool(s, nv, vis.size + 5, pool)
    assert np.array_equal(got[: vis.size], vis) and np.all(got[vis.size:] == -1)


def test_reindex_pool_mode_searches_the_full_selection_pool():
    """index_topk(REINDEX_POOL, prev_idx = the FULL selection) = per-query top-K over the pool
    of that query's FULL selection; plain REINDEX scans every visible entry, prev_idx or not."""
    rng = np.random.default_rng(6)
    T, H_I, N, K = 3, 2, 256, 16
    q = rng.standard_normal((T, H_I, 64)); w = np.abs(rng.standard_normal((T, H_I)))
    z = rng.standard_normal((N, 64)); nv = np.array([256, 200, 31])
    full = indexer.index_topk(0, q, w, z, nv, K)
    q2 = rng.standard_normal((T, H_I, 64)); z2 = rng.standard_normal((N, 64))
    got = indexer.index_topk(3, q2, w, z2, nv, K, prev_idx=full)
    I = indexer.scores(q2, w, z2)
    for t in range(T):
        assert np.array_equal(got[t], indexer.topk_in_pool(I[t], nv[t], K, indexer.candidate_pool(full[t])))
    full_scan = np.stack([indexer.topk(I[t], nv[t], K) for t in range(T)])
    assert np.array_equal(indexer.index_topk(1, q2, w, z2, nv, K), full_scan)
    assert np.array_equal(indexer.index_topk(1, q2, w, z2, nv, K, prev_idx=full), full_scan)
