"""Indexer + top-K parity: CUDA index sets equal the oracle's up to ties within 1e-6
relative of the K-th score; exact when the arithmetic is exact (integer data).

Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", picx.dev summary,
Methodology / 2. CSA2 (FULL / REINDEX compute fresh top-K, REUSE repeats them).
"""
import numpy as np
import pytest
import torch

import csa2_inputs as ci
import sparse_attention_kv_decode_b300 as csa2
from oracle import indexer
from tests._util import check_index_set, f64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _run(q_bits, w, z_bits, nvis, K, mode=csa2.FULL, with_scores=True):
    B, T, H_I, _ = q_bits.shape
    dev = "cuda"
    out_s = torch.empty((B, T, K), dtype=torch.float32, device=dev) if with_scores else None
    idx = csa2.csa2_index_topk(mode, to_dev_bf16(q_bits, dev), to_dev(w, dev), to_dev_bf16(z_bits, dev),
                               to_dev(nvis.astype(np.int32), dev), K, out_scores=out_s)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), (out_s.cpu().numpy() if with_scores else None)


def _check_all(q_bits, w, z_bits, nvis, K):
    B, T = q_bits.shape[:2]
    got, gs = _run(q_bits, w, z_bits, nvis, K)
    ndiff = 0
    for b in range(B):
        I = indexer.scores(f64(q_bits[b]), w[b], f64(z_bits[b]))
        for t in range(T):
            nv = int(nvis[b * T + t])
            want = indexer.topk(I[t], nv, K)
            ndiff += check_index_set(got[b, t], want, I[t], nv, K)
            sel = got[b, t][got[b, t] >= 0]
            # returned scores are the fp32 scores of the returned indices
            np.testing.assert_allclose(gs[b, t, :sel.size], I[t][sel], rtol=2e-5, atol=2e-5)
            assert np.all(np.isnan(gs[b, t, sel.size:]))
    return got, ndiff


def test_tiny_config():
    cfg = ci.TINY
    inp = ci.make_decode_inputs(cfg, with_x=False)
    L = inp.layers[0]
    _check_all(L.q_idx, L.w_idx, L.z, inp.n_visible, cfg.K)


@pytest.mark.parametrize("N,K,H_I", [(4096, 512, 8), (3000, 256, 4), (5000, 2048, 16), (1, 4, 3), (700, 700, 8),
                                     (9000, 4096, 8)])
def test_scaled_decode_shapes(N, K, H_I):
    cfg = ci.scaled(ci.DECODE_128K, B=3, N=N, H=16, H_I=H_I, K=K, W=8, modes=(ci.FULL,))
    inp = ci.make_decode_inputs(cfg, with_x=False)
    L = inp.layers[0]
    _check_all(L.q_idx, L.w_idx, L.z, inp.n_visible, K)


def test_causal_visibility_and_padding():
    rng = np.random.default_rng(21)
    B, T, N, H_I, K = 2, 5, 2000, 8, 300
    q = ci.bf16_bits(rng.standard_normal((B, T, H_I, 64), dtype=np.float32))
    w = np.abs(rng.standard_normal((B, T, H_I), dtype=np.float32))
    z = ci.bf16_bits(rng.standard_normal((B, N, 64), dtype=np.float32))
    nvis = np.array([0, 1, 299, 300, 301, 2000, 1999, 5, 1024, 1500], dtype=np.int32)
    _check_all(q, w, z, nvis, K)


@pytest.mark.parametrize("B,T,N,H_I,K", [(2, 100, 5000, 8, 512), (1, 40, 3000, 16, 300), (3, 70, 1500, 4, 200),
                                          (1, 300, 9000, 8, 2048)])
def test_many_query_tokens_gemm_scoring(B, T, N, H_I, K):
    """Query tokens in tiles of 256 / H_I scored as one keys x (token, head) GEMM on the
    tensor cores (a partial last tile, ragged causal limits including 0 and N, key tiles
    past a tile's largest limit skipped): sets and returned scores match the oracle."""
    rng = np.random.default_rng(25 + T)
    q = ci.bf16_bits(rng.standard_normal((B, T, H_I, 64), dtype=np.float32))
    w = np.abs(rng.standard_normal((B, T, H_I), dtype=np.float32))
    z = ci.bf16_bits(rng.standard_normal((B, N, 64), dtype=np.float32))
    nvis = rng.integers(0, N + 1, B * T).astype(np.int32)
    nvis[0], nvis[-1], nvis[1] = 0, N, N - 1
    _check_all(q, w, z, nvis, K)


def test_exact_ties_resolved_to_lower_index():
    """Small integers make every dot product exact in fp32 and fp64, so scores tie
    exactly and the selection must equal the oracle's with no tolerance."""
    rng = np.random.default_rng(22)
    B, T, N, H_I, K = 2, 2, 9000, 8, 1000
    q = ci.bf16_bits(rng.integers(-2, 3, (B, T, H_I, 64)).astype(np.float32))
    w = rng.integers(0, 3, (B, T, H_I)).astype(np.float32)
    z = ci.bf16_bits(rng.integers(-1, 2, (B, N, 64)).astype(np.float32))
    nvis = np.array([N, 7000, N, 4321], dtype=np.int32)
    got, _ = _run(q, w, z, nvis, K)
    for b in range(B):
        I = indexer.scores(f64(q[b]), w[b], f64(z[b]))
        for t in range(T):
            assert np.array_equal(got[b, t], indexer.topk(I[t], nvis[b * T + t], K))


@pytest.mark.parametrize("levels", [128, 16])
def test_clustered_scores_need_refinement(levels):
    """Exact scores (one head, q = e_0, w = 1: the score is z[n, 0]) packed into a narrow band
    1 + j/128 (j < levels) with one far outlier (2^100): the first histogram round puts the
    whole band in one bin, the next one bins the band exactly; with 16 levels every level
    repeats ~375 times, so the K-th score's bin is all ties (lowest positions first)."""
    B, T, N, H_I, K = 1, 2, 6000, 8, 3000
    q = np.zeros((B, T, H_I, 64), np.float32)
    q[..., 0, 0] = 1.0
    w = np.zeros((B, T, H_I), np.float32)
    w[..., 0] = 1.0
    z = np.zeros((B, N, 64), np.float32)
    z[0, :, 0] = 1.0 + (np.arange(N) % levels) / 128.0
    z[0, 4321, 0] = 2.0 ** 100
    zb, qb = ci.bf16_bits(z), ci.bf16_bits(q)
    nvis = np.array([N, N - 1], np.int32)
    got, _ = _run(qb, w, zb, nvis, K)
    I = indexer.scores(f64(qb[0]), w[0], f64(zb[0]))
    for t in range(T):
        assert np.array_equal(got[0, t], indexer.topk(I[t], nvis[t], K))


def test_all_scores_equal():
    B, T, N, H_I, K = 1, 1, 5000, 8, 777
    q = np.zeros((B, T, H_I, 64), np.uint16)
    w = np.ones((B, T, H_I), np.float32)
    z = ci.bf16_bits(np.random.default_rng(23).standard_normal((B, N, 64), dtype=np.float32))
    got, _ = _run(q, w, z, np.array([N], np.int32), K)
    assert np.array_equal(got[0, 0], np.arange(K))


def test_k_at_least_visible_selects_all():
    rng = np.random.default_rng(24)
    q = ci.bf16_bits(rng.standard_normal((1, 1, 8, 64), dtype=np.float32))
    w = np.abs(rng.standard_normal((1, 1, 8), dtype=np.float32))
    z = ci.bf16_bits(rng.standard_normal((1, 600, 64), dtype=np.float32))
    got, _ = _run(q, w, z, np.array([600], np.int32), 1024)
    assert np.array_equal(got[0, 0, :600], np.arange(600)) and np.all(got[0, 0, 600:] == -1)


def test_full_size_decode_128k_layer():
    """32 sequences x 32768 entries, K = 2048, the planted recency bias: all 32 queries."""
    cfg = ci.scaled(ci.DECODE_128K, modes=(ci.FULL,))
    inp = ci.make_decode_inputs(cfg, with_x=False)
    L = inp.layers[0]
    _, ndiff = _check_all(L.q_idx, L.w_idx, L.z, inp.n_visible, cfg.K)
    print("tie-band differences:", ndiff)


def test_full_size_decode_1m():
    """4 sequences x 262144 entries (16-CTA clusters), K = 2048."""
    cfg = ci.DECODE_1M
    inp = ci.make_decode_inputs(cfg, with_x=False)
    L = inp.layers[0]
    _check_all(L.q_idx, L.w_idx, L.z, inp.n_visible, cfg.K)


def test_reuse_copies_and_aliases():
    prev = torch.arange(3 * 2 * 16, dtype=torch.int32, device="cuda").reshape(3, 2, 16)
    out = torch.full_like(prev, -7)
    r = csa2.csa2_index_topk(csa2.REUSE, None, None, None, None, 16, prev_idx=prev, out_idx=out)
    torch.cuda.synchronize()
    assert torch.equal(r, prev) and torch.equal(out, prev)
    same = csa2.csa2_index_topk(csa2.REUSE, None, None, None, None, 16, prev_idx=prev, out_idx=prev)
    assert torch.equal(same, prev)


@pytest.mark.parametrize("B,N", [(6, 20000), (3, 40000), (33, 4099)])
def test_warp_runs_across_query_boundaries(B, N):
    """All entries visible, at sizes where a scoring CTA's run of key-group chunks ends
    inside one query and continues in the next (the chunks are split evenly over 296 CTAs,
    not per query, and a CTA's warps take them in turn): every query's last groups must be
    scored with that query's indexer rows."""
    cfg = ci.scaled(ci.DECODE_128K, B=B, N=N, H=16, K=256, W=8, modes=(ci.FULL,))
    inp = ci.make_decode_inputs(cfg, with_x=False)
    L = inp.layers[0]
    _check_all(L.q_idx, L.w_idx, L.z, np.full(B, N, np.int32), cfg.K)


@pytest.mark.parametrize("B,N,H_I", [(45, 4111, 8), (70, 1000, 8), (19, 4111, 16)])
def test_scoring_chunks_with_ragged_single_tokens(B, N, H_I):
    """One token per sequence with ragged visible counts (0, 1, group and chunk edges,
    full) and an odd number of 16-key groups per query, so that each query's last chunk
    holds one group and chunk runs end inside queries: every query must be scored over
    exactly its visible entries with its own indexer rows and weights."""
    rng = np.random.default_rng(2000 + B + N + H_I)
    K = 200
    q = ci.bf16_bits(rng.standard_normal((B, 1, H_I, 64), dtype=np.float32))
    w = np.abs(rng.standard_normal((B, 1, H_I), dtype=np.float32))
    z = ci.bf16_bits(rng.standard_normal((B, N, 64), dtype=np.float32))
    edges = np.array([0, 1, 15, 16, 17, 31, 32, 33, 200, 201, N - 1, N], dtype=np.int32)
    nvis = np.where(rng.random(B) < 0.5, edges[rng.integers(0, edges.size, B)],
                    rng.integers(0, N + 1, B)).astype(np.int32)
    _check_all(q, w, z, nvis, K)


@pytest.mark.parametrize("B,T,H_I", [(40, 2, 8), (37, 3, 4), (9, 5, 8), (21, 3, 8), (12, 2, 16)])
def test_decode_key_tiles_split_over_ctas_ragged(B, T, H_I):
    """A few query tokens per sequence (the N = 16 tensor-core scoring for H_I = 4, 8),
    ragged visible counts (0, 1, tile edges, full):
    the key tiles each (sequence, token tile) needs are counted on the device and split
    evenly over the CTAs, so a CTA's run starts and ends inside sequences and token
    tiles; every query must get its own keys, indexer rows and weights."""
    rng = np.random.default_rng(1000 + B * T * H_I)
    N, K = 3000, 200
    q = ci.bf16_bits(rng.standard_normal((B, T, H_I, 64), dtype=np.float32))
    w = np.abs(rng.standard_normal((B, T, H_I), dtype=np.float32))
    z = ci.bf16_bits(rng.standard_normal((B, N, 64), dtype=np.float32))
    edges = np.array([0, 1, 127, 128, 129, 200, 201, 2999, 3000, 1500], dtype=np.int32)
    nvis = np.where(rng.random(B * T) < 0.5, edges[rng.integers(0, edges.size, B * T)],
                    rng.integers(0, N + 1, B * T)).astype(np.int32)
    _check_all(q, w, z, nvis, K)


def test_deterministic_repeat():
    cfg = ci.scaled(ci.DECODE_128K, B=4, N=8192, K=1024, modes=(ci.FULL,))
    inp = ci.make_decode_inputs(cfg, with_x=False)
    L = inp.layers[0]
    a, _ = _run(L.q_idx, L.w_idx, L.z, inp.n_visible, cfg.K)
    b, _ = _run(L.q_idx, L.w_idx, L.z, inp.n_visible, cfg.K)
    assert np.array_equal(a, b)


# ---- REINDEX over the candidate pool (Hierarchical Sparse Indexer, picx.dev summary,
# Methodology / 3): the pool is built from the GPU's own FULL selection, and the oracle
# ranks the same pool's visible positions.

def _check_pool(L_full, L_re, nvis, K, exact=False):
    B, T = L_re.q_idx.shape[:2]
    dev = "cuda"
    full, _ = _run(L_full.q_idx, L_full.w_idx, L_full.z, nvis, K, with_scores=False)
    out_s = torch.empty((B, T, K), dtype=torch.float32, device=dev)
    got = csa2.csa2_index_topk(csa2.REINDEX_POOL, to_dev_bf16(L_re.q_idx, dev), to_dev(L_re.w_idx, dev),
                               to_dev_bf16(L_re.z, dev), to_dev(nvis.astype(np.int32), dev), K,
                               prev_idx=torch.from_numpy(full).to(dev), out_scores=out_s)
    torch.cuda.synchronize()
    got, gs = got.cpu().numpy(), out_s.cpu().numpy()
    ndiff = 0
    for b in range(B):
        I = indexer.scores(f64(L_re.q_idx[b]), L_re.w_idx[b], f64(L_re.z[b]))
        for t in range(T):
            nv = int(nvis[b * T + t])
            pool = indexer.candidate_pool(full[b, t])
            vis = pool[pool < nv]
            want = indexer.topk_in_pool(I[t], nv, K, pool)
            g = got[b, t][got[b, t] >= 0]
            assert np.all(np.diff(g) > 0) and g.size == min(K, vis.size)
            assert np.all(got[b, t][g.size:] == -1)
            assert np.all(np.isin(g, vis)), "selected outside the pool"
            if exact:
                assert np.array_equal(got[b, t], want)
            else:
                s = np.sort(I[t][vis])[::-1]
                kth = s[K - 1] if K <= s.size else -np.inf
                diff = np.setxor1d(g, want[want >= 0])
                if diff.size:
                    bad = diff[np.abs(I[t][diff] - kth) > 1e-6 * abs(kth)]
                    assert bad.size == 0, f"{bad.size} pool-set differences outside the tie band"
                ndiff += diff.size
            np.testing.assert_allclose(gs[b, t, :g.size], I[t][g], rtol=2e-5, atol=2e-5)
    return ndiff


@pytest.mark.parametrize("N,K", [(4096, 256), (3001, 300), (20000, 1024)])
def test_reindex_pool_scaled(N, K):
    cfg = ci.scaled(ci.DECODE_128K, B=3, N=N, H=16, K=K, W=8, modes=(ci.FULL, ci.REINDEX))
    inp = ci.make_decode_inputs(cfg, with_x=False)
    _check_pool(inp.layers[0], inp.layers[1], inp.n_visible, K)


def test_reindex_pool_causal_ragged():
    """Several query tokens per sequence with ragged visibility (partial last blocks, fewer
    visible pool positions than K, a single visible entry)."""
    cfg = ci.scaled(ci.PREFILL_CHUNK, B=2, T=6, N=3000, H=16, K=200, W=8, modes=(ci.FULL, ci.REINDEX))
    inp = ci.make_decode_inputs(cfg, with_x=False)
    nvis = np.array([1, 7, 9, 200, 1603, 3000, 2999, 8, 16, 17, 640, 2048], dtype=np.int32)
    _check_pool(inp.layers[0], inp.layers[1], nvis, cfg.K)


def test_reindex_pool_many_query_tokens():
    """2100 query tokens of one sequence over a short cache (640 entries, pools of one to
    eight blocks per token, causal): warp runs of the pooled scoring cross many queries."""
    cfg = ci.scaled(ci.PREFILL_CHUNK, B=1, T=2100, N=640, H=16, K=64, W=8, modes=(ci.FULL, ci.REINDEX))
    inp = ci.make_decode_inputs(cfg, with_x=False)
    _check_pool(inp.layers[0], inp.layers[1], inp.n_visible, cfg.K)


def test_reindex_pool_exact_ties():
    """Integer data: exact scores and ties, so the pool selection must equal the oracle's."""
    rng = np.random.default_rng(31)
    B, T, N, H_I, K = 2, 2, 9000, 8, 700

    class L:
        pass
    Lf, Lr = L(), L()
    for Lx in (Lf, Lr):
        Lx.q_idx = ci.bf16_bits(rng.integers(-2, 3, (B, T, H_I, 64)).astype(np.float32))
        Lx.w_idx = rng.integers(0, 3, (B, T, H_I)).astype(np.float32)
        Lx.z = ci.bf16_bits(rng.integers(-1, 2, (B, N, 64)).astype(np.float32))
    _check_pool(Lf, Lr, np.array([N, 7000, 5555, 4321], dtype=np.int32), K, exact=True)


def test_reindex_pool_full_size_128k():
    """32 sequences x 32768 entries, K = 2048: REINDEX ranks at most 16,384 pool positions."""
    cfg = ci.scaled(ci.DECODE_128K, modes=(ci.FULL, ci.REINDEX))
    inp = ci.make_decode_inputs(cfg, with_x=False)
    _check_pool(inp.layers[0], inp.layers[1], inp.n_visible, cfg.K)


def test_reindex_pool_full_size_1m():
    """4 sequences x 262144 entries: the pool keeps REINDEX at <= 16,384 positions."""
    cfg = ci.scaled(ci.DECODE_1M, modes=(ci.FULL, ci.REINDEX))
    inp = ci.make_decode_inputs(cfg, with_x=False)
    _check_pool(inp.layers[0], inp.layers[1], inp.n_visible, cfg.K)


def test_reindex_pool_flags_a_selection_out_of_order():
    """prev_idx that is not ascending, or holds an index past the cache, sets the device
    bad-index bit; the call still completes with in-range indices."""
    rng = np.random.default_rng(32)
    B, T, N, H_I, K = 1, 2, 2048, 8, 64
    q = ci.bf16_bits(rng.standard_normal((B, T, H_I, 64), dtype=np.float32))
    w = np.abs(rng.standard_normal((B, T, H_I), dtype=np.float32))
    z = ci.bf16_bits(rng.standard_normal((B, N, 64), dtype=np.float32))
    prev = np.sort(rng.choice(N, size=(B, T, K)), axis=-1).astype(np.int32)
    prev[0, 0, 5], prev[0, 0, 6] = prev[0, 0, 6] + 1, prev[0, 0, 5]   # out of order
    prev[0, 1, -1] = N + 100                                           # past the cache
    dev = "cuda"
    ws = csa2.csa2_workspace(B, T, 0, N, K, device=dev)
    got = csa2.csa2_index_topk(csa2.REINDEX_POOL, to_dev_bf16(q, dev), to_dev(w, dev), to_dev_bf16(z, dev),
                               to_dev(np.full(B * T, N, np.int32), dev), K, prev_idx=torch.from_numpy(prev).to(dev),
                               ws=ws)
    st, flags = csa2.csa2_read_device_status(ws)
    assert flags & csa2.DEV_BAD_INDEX
    g = got.cpu().numpy()
    assert np.all((g == -1) | ((g >= 0) & (g < N)))
