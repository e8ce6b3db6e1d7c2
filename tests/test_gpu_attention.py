"""Sparse decode + SWA merge parity against the FP64 oracle (max-abs 2e-3, rel-L2 1e-3),
through the separate calls (csa2_index_topk, csa2_sparse_decode, csa2_swa_merge) and
through the one-layer call (csa2_decode_layer: the selection, then csa2_decode_attention).

Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression": sparse attention
over the whole context combined with a sliding-window branch (blog repost), the CSA2
layer modes and the FP4 main KV (picx.dev summary, Methodology / 2 and / 5).
The oracle attends over the GPU's own index set (which may differ from the oracle's only
inside the top-K tie band, checked separately).
"""
import numpy as np
import pytest
import torch

import csa2_inputs as ci
import sparse_attention_kv_decode_b300 as csa2
from oracle import attention, fp4, indexer
from tests._util import check_attention, check_index_set, check_lse, f64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _cache(X):
    codes, scales = csa2.csa2_encode_kv(to_dev(X, DEV))
    return codes, scales


def _oracle_query(q_bits_bt, rows_of, idx, swa_bits_b, ws, wl, cfg):
    """Oracle global branch over idx, SWA branch, merge. rows_of(idx array) -> dequantised rows."""
    q = f64(q_bits_bt)
    sel = idx[idx >= 0]
    og, lg = attention.attend(q, rows_of(sel), cfg.d_v, cfg.softmax_scale)
    os_, ls = attention.swa_branch(q, f64(swa_bits_b), int(ws), int(wl), cfg.d_v, cfg.softmax_scale)
    O, L = attention.merge(og, lg, os_, ls)
    return og, lg, O, L


def _run_group(cfg, inp, sample=None, fused=True, t_sample=None):
    """Run every layer of the group on the GPU; compare (sampled) sequences and query tokens
    with the oracle."""
    B, T = cfg.B, cfg.T
    ws = csa2.csa2_workspace(B, T, cfg.H, cfg.N, cfg.K, device=DEV)
    nvis = to_dev(inp.n_visible, DEV)
    wst, wln = to_dev(inp.win_start, DEV), to_dev(inp.win_len, DEV)
    codes = scales = None
    prev = None
    kv_host = {}
    results = []
    for li, L in enumerate(inp.layers):
        if L.mode == ci.FULL:
            codes, scales = _cache(L.X)
            kv_host = dict(X=L.X)
        before = (codes.clone(), scales.clone()) if L.mode != ci.FULL else None
        qd = to_dev_bf16(L.q, DEV)
        kw = {}
        if L.mode != ci.REUSE:
            kw = dict(q_idx=to_dev_bf16(L.q_idx, DEV), w_idx=to_dev(L.w_idx, DEV), z=to_dev_bf16(L.z, DEV),
                      n_visible=nvis)
        o, lse, idx = csa2.decode_layer(L.mode, qd, codes, scales, to_dev_bf16(L.swa, DEV), wst, wln, cfg.W,
                                        cfg.K, prev_idx=prev, ws=ws, fused=fused, **kw)
        torch.cuda.synchronize()
        st, flags = csa2.csa2_read_device_status(ws)
        assert st == 0, (st, flags)
        if before is not None:   # REINDEX / REUSE leave the main KV untouched
            assert torch.equal(before[0], codes) and torch.equal(before[1], scales)
        idx_h = idx.cpu().numpy()
        if L.mode == ci.REUSE:
            assert np.array_equal(idx_h, prev.cpu().numpy())
        results.append((L, o.cpu().numpy(), lse.cpu().numpy(), idx_h))
        prev = idx

    bs = range(B) if sample is None else sample
    ts = list(range(T)) if t_sample is None else list(t_sample)
    X = kv_host["X"]
    for b in bs:
        cache_rows = {}

        def rows_of(sel, b=b):
            out = np.empty((sel.size, 576))
            miss = [i for i in sel.tolist() if i not in cache_rows]
            if miss:
                miss = np.array(sorted(set(miss)))
                dq = fp4.decode(*fp4.encode(X[b, miss]))
                for i, r in zip(miss.tolist(), dq):
                    cache_rows[i] = r
            for k, i in enumerate(sel.tolist()):
                out[k] = cache_rows[i]
            return out

        for (L, o, lse, idx_h) in results:
            if L.mode != ci.REUSE:
                I = dict(zip(ts, indexer.scores(f64(L.q_idx[b][ts]), L.w_idx[b][ts], f64(L.z[b]))))
            for t in ts:
                qi = b * T + t
                if L.mode != ci.REUSE:
                    want = indexer.topk(I[t], inp.n_visible[qi], cfg.K)
                    check_index_set(idx_h[b, t], want, I[t], inp.n_visible[qi], cfg.K)
                _, _, O, LSE = _oracle_query(L.q[b, t], rows_of, idx_h[b, t], L.swa[b], inp.win_start[qi],
                                             inp.win_len[qi], cfg)
                check_attention(o[b, t], O, f"layer {ci.MODE_NAMES[L.mode]} b={b} t={t}")
                check_lse(lse[b, t], LSE, f"layer {ci.MODE_NAMES[L.mode]} b={b} t={t}")
    return results


@pytest.mark.parametrize("fused", [True, False])
def test_tiny_config_layer(fused):
    _run_group(ci.TINY, ci.make_decode_inputs(ci.TINY), fused=fused)


@pytest.mark.parametrize("fused", [True, False])
def test_scaled_group_full_reindex_reuse(fused):
    cfg = ci.scaled(ci.DECODE_128K, B=3, N=4096, K=512)
    _run_group(cfg, ci.make_decode_inputs(cfg), fused=fused)


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("H,K,W", [(16, 200, 100), (32, 1000, 1), (48, 64, 256), (64, 130, 0), (64, 2048, 200),
                                   (64, 4096, 256)])
def test_ragged_shapes(H, K, W, fused):
    """Head counts 16-64, K from 64 to the largest supported (4096), windows from none to
    the largest (256 rows)."""
    N = 5000 if K > 2048 else 2500
    cfg = ci.scaled(ci.DECODE_128K, B=2, N=N, H=H, K=K, W=max(W, 1), modes=(ci.FULL, ci.REUSE))
    inp = ci.make_decode_inputs(cfg)
    if W == 0:
        inp.win_len[:] = 0
    _run_group(cfg, inp, fused=fused)


@pytest.mark.parametrize("fused", [True, False])
def test_prefill_like_many_queries_causal(fused):
    cfg = ci.scaled(ci.PREFILL_CHUNK, T=37, N=1200, K=256, W=16)
    _run_group(cfg, ci.make_decode_inputs(cfg), fused=fused)


def test_global_equals_dense_when_k_covers_all():
    cfg = ci.scaled(ci.TINY, N=300, K=512, H=32, W=8)
    inp = ci.make_decode_inputs(cfg)
    L = inp.layers[0]
    codes, scales = _cache(L.X)
    idx = torch.from_numpy(np.tile(np.concatenate([np.arange(300), -np.ones(212)]).astype(np.int32),
                                   (1, 1, 1))).to(DEV)
    o, lse = csa2.csa2_sparse_decode(to_dev_bf16(L.q, DEV), codes, scales, idx, cfg.softmax_scale)
    torch.cuda.synchronize()
    rows = fp4.decode(*fp4.encode(L.X[0]))
    O, LSE = attention.attend(f64(L.q[0, 0]), rows, 512, cfg.softmax_scale)
    check_attention(o[0, 0].cpu().numpy(), O, "dense")
    check_lse(lse[0, 0].cpu().numpy(), LSE, "dense")


def test_empty_selection_and_pure_swa():
    cfg = ci.scaled(ci.TINY, N=64, K=64, H=16, W=32)
    inp = ci.make_decode_inputs(cfg)
    L = inp.layers[0]
    codes, scales = _cache(L.X)
    idx = torch.full((1, 1, 64), -1, dtype=torch.int32, device=DEV)
    q = to_dev_bf16(L.q, DEV)
    o_g, lse_g = csa2.csa2_sparse_decode(q, codes, scales, idx, cfg.softmax_scale)
    o, lse = csa2.csa2_swa_merge(q, to_dev_bf16(L.swa, DEV), to_dev(inp.win_start, DEV), to_dev(inp.win_len, DEV),
                                 cfg.W, o_g, lse_g, cfg.softmax_scale)
    torch.cuda.synchronize()
    assert torch.all(o_g == 0) and torch.all(torch.isneginf(lse_g))
    O, LSE = attention.swa_branch(f64(L.q[0, 0]), f64(L.swa[0]), 0, cfg.W, 512, cfg.softmax_scale)
    check_attention(o[0, 0].cpu().numpy(), O, "swa only")
    # both branches empty
    o2, lse2 = csa2.csa2_swa_merge(q, to_dev_bf16(L.swa, DEV), to_dev(inp.win_start, DEV),
                                   torch.zeros(1, dtype=torch.int32, device=DEV), cfg.W, o_g, lse_g)
    torch.cuda.synchronize()
    assert torch.all(o2 == 0) and torch.all(torch.isneginf(lse2))


def test_fused_empty_branches():
    """One call over an empty selection and/or an empty window."""
    cfg = ci.scaled(ci.TINY, N=64, K=64, H=16, W=32)
    inp = ci.make_decode_inputs(cfg)
    L = inp.layers[0]
    codes, scales = _cache(L.X)
    q = to_dev_bf16(L.q, DEV)
    swa = to_dev_bf16(L.swa, DEV)
    wst = to_dev(inp.win_start, DEV)
    none = torch.full((1, 1, 64), -1, dtype=torch.int32, device=DEV)
    allk = torch.arange(64, dtype=torch.int32, device=DEV).reshape(1, 1, 64)
    zero = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, lse = csa2.csa2_decode_attention(q, codes, scales, none, swa, wst, to_dev(inp.win_len, DEV), cfg.W,
                                        cfg.softmax_scale)
    torch.cuda.synchronize()
    O, LSE = attention.swa_branch(f64(L.q[0, 0]), f64(L.swa[0]), 0, cfg.W, 512, cfg.softmax_scale)
    check_attention(o[0, 0].cpu().numpy(), O, "window only")
    check_lse(lse[0, 0].cpu().numpy(), LSE, "window only")
    o, lse = csa2.csa2_decode_attention(q, codes, scales, allk, swa, wst, zero, cfg.W, cfg.softmax_scale)
    torch.cuda.synchronize()
    rows = fp4.decode(*fp4.encode(L.X[0]))
    O, LSE = attention.attend(f64(L.q[0, 0]), rows, 512, cfg.softmax_scale)
    check_attention(o[0, 0].cpu().numpy(), O, "entries only")
    check_lse(lse[0, 0].cpu().numpy(), LSE, "entries only")
    o, lse = csa2.csa2_decode_attention(q, codes, scales, none, swa, wst, zero, cfg.W, cfg.softmax_scale)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_fused_window_rows_past_the_window_are_ignored():
    """NaN rows right after the window (inside the same 128-row tile) must not leak into O."""
    cfg = ci.scaled(ci.TINY, N=64, K=64, H=16, W=40)
    inp = ci.make_decode_inputs(cfg)
    L = inp.layers[0]
    codes, scales = _cache(L.X)
    S = 128
    swa_bits = np.full((1, S, 576), 0x7FC0, dtype=np.uint16)   # bf16 NaN after the 40 window rows
    swa_bits[0, :40] = L.swa[0, :40]
    idx = torch.arange(64, dtype=torch.int32, device=DEV).reshape(1, 1, 64)
    o, lse = csa2.csa2_decode_attention(to_dev_bf16(L.q, DEV), codes, scales, idx, to_dev_bf16(swa_bits, DEV),
                                        torch.zeros(1, dtype=torch.int32, device=DEV),
                                        torch.tensor([40], dtype=torch.int32, device=DEV), cfg.W,
                                        cfg.softmax_scale)
    torch.cuda.synchronize()
    assert S > 40
    rows = fp4.decode(*fp4.encode(L.X[0]))
    og, lg = attention.attend(f64(L.q[0, 0]), rows, 512, cfg.softmax_scale)
    os_, ls = attention.swa_branch(f64(L.q[0, 0]), f64(L.swa[0]), 0, 40, 512, cfg.softmax_scale)
    O, LSE = attention.merge(og, lg, os_, ls)
    check_attention(o[0, 0].cpu().numpy(), O, "fused, NaN past window")
    check_lse(lse[0, 0].cpu().numpy(), LSE, "fused, NaN past window")


def test_device_checks_flag_bad_index_and_window():
    cfg = ci.scaled(ci.TINY, N=64, K=64, H=16, W=32)
    inp = ci.make_decode_inputs(cfg)
    L = inp.layers[0]
    codes, scales = _cache(L.X)
    ws = csa2.csa2_workspace(1, 1, 16, 64, 64, device=DEV)
    idx = torch.arange(64, dtype=torch.int32, device=DEV).reshape(1, 1, 64).clone()
    idx[0, 0, 5] = 64          # outside the cache: skipped and flagged
    idx[0, 0, 6] = -9
    q = to_dev_bf16(L.q, DEV)
    o_g, lse_g = csa2.csa2_sparse_decode(q, codes, scales, idx, cfg.softmax_scale, ws=ws)
    st, flags = csa2.csa2_read_device_status(ws)
    assert st == 6 and flags & csa2.DEV_BAD_INDEX
    keep = np.array([i for i in range(64) if i not in (5, 6)])
    rows = fp4.decode(*fp4.encode(L.X[0]))
    O, _ = attention.attend(f64(L.q[0, 0]), rows[keep], 512, cfg.softmax_scale)
    check_attention(o_g[0, 0].cpu().numpy(), O, "bad index skipped")
    st, flags = csa2.csa2_read_device_status(ws)
    assert st == 0 and flags == 0
    csa2.csa2_swa_merge(q, to_dev_bf16(L.swa, DEV), torch.tensor([20], dtype=torch.int32, device=DEV),
                        torch.tensor([32], dtype=torch.int32, device=DEV), cfg.W, o_g, lse_g, ws=ws)
    st, flags = csa2.csa2_read_device_status(ws)
    assert st == 6 and flags & csa2.DEV_BAD_WINDOW


def test_full_size_decode_128k_group_sampled():
    """The bench workload: 32 x 32768 entries, 64 heads, K = 2048, FULL -> REINDEX -> REUSE,
    in the bench's launch configuration (fused attention); 3 sequences checked against the oracle."""
    cfg = ci.DECODE_128K
    _run_group(cfg, ci.make_decode_inputs(cfg), sample=[0, 17, 31])


def test_full_size_decode_1m_sampled():
    """4 sequences over 262,144 entries each (1M tokens at 4:1), K = 2048, one FULL layer: the
    four queries split 16 ways (16-CTA clusters, the merge for more than four splits);
    sequences 0 and 3 checked against the oracle."""
    cfg = ci.DECODE_1M
    _run_group(cfg, ci.make_decode_inputs(cfg), sample=[0, 3])


def test_full_size_prefill_chunk_sampled():
    """4096 query tokens of one sequence over 32768 entries with causal visibility, K = 2048,
    window 128 (the prefill-chunk workload); first, middle and last tokens checked."""
    cfg = ci.PREFILL_CHUNK
    _run_group(cfg, ci.make_decode_inputs(cfg), t_sample=[0, 1, 777, 2048, 4095])


def test_full_size_decode_128k_two_calls_sampled():
    cfg = ci.DECODE_128K
    _run_group(cfg, ci.make_decode_inputs(cfg), sample=[5], fused=False)


def test_deterministic_outputs():
    cfg = ci.scaled(ci.DECODE_128K, B=2, N=2048, K=256, modes=(ci.FULL,))
    inp = ci.make_decode_inputs(cfg)
    a = _run_group(cfg, inp)
    b = _run_group(cfg, inp)
    for (_, oa, la, ia), (_, ob, lb, ib) in zip(a, b):
        assert np.array_equal(oa, ob) and np.array_equal(la, lb) and np.array_equal(ia, ib)


def test_decode_layer_equals_topk_then_attention():
    """csa2_decode_layer (whose selection also requests the selected FP4 rows into L2) writes
    exactly what csa2_index_topk followed by csa2_decode_attention writes."""
    cfg = ci.scaled(ci.DECODE_128K, B=4, N=4096, K=512)
    inp = ci.make_decode_inputs(cfg)
    B, T = cfg.B, cfg.T
    ws = csa2.csa2_workspace(B, T, cfg.H, cfg.N, cfg.K, device=DEV)
    nvis = to_dev(inp.n_visible, DEV)
    wst, wln = to_dev(inp.win_start, DEV), to_dev(inp.win_len, DEV)
    prev = None
    codes = scales = None
    for L in inp.layers:
        if L.mode == ci.FULL:
            codes, scales = _cache(L.X)
        qd, swa = to_dev_bf16(L.q, DEV), to_dev_bf16(L.swa, DEV)
        kw = {}
        if L.mode != ci.REUSE:
            kw = dict(q_idx=to_dev_bf16(L.q_idx, DEV), w_idx=to_dev(L.w_idx, DEV), z=to_dev_bf16(L.z, DEV),
                      n_visible=nvis)
        o1, l1, i1 = csa2.csa2_decode_layer(L.mode, qd, codes, scales, swa, wst, wln, cfg.W, cfg.K,
                                            prev_idx=prev, ws=ws, **kw)
        i2 = csa2.csa2_index_topk(L.mode, kw.get("q_idx"), kw.get("w_idx"), kw.get("z"), kw.get("n_visible"),
                                  cfg.K, prev_idx=prev, out_idx=torch.empty_like(i1), ws=ws)
        o2, l2 = csa2.csa2_decode_attention(qd, codes, scales, i2, swa, wst, wln, cfg.W, ws=ws)
        torch.cuda.synchronize()
        assert csa2.csa2_read_device_status(ws)[0] == 0
        assert torch.equal(i1, i2)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        prev = i1


def test_range_flag_for_values_outside_fp16():
    """The products run on fp16 tensor cores: a bf16 query or window value above 65504 in
    magnitude sets CSA2_DEV_RANGE; 65280 (the largest bf16 value below it) does not."""
    cfg = ci.scaled(ci.TINY, N=64, K=64, H=16, W=32)
    inp = ci.make_decode_inputs(cfg)
    L = inp.layers[0]
    codes, scales = _cache(L.X)
    ws = csa2.csa2_workspace(1, 1, 16, 64, 64, device=DEV)
    idx = torch.arange(64, dtype=torch.int32, device=DEV).reshape(1, 1, 64)
    wst, wln = to_dev(inp.win_start, DEV), to_dev(inp.win_len, DEV)

    def run(q_bits, swa_bits):
        csa2.csa2_decode_attention(to_dev_bf16(q_bits, DEV), codes, scales, idx, to_dev_bf16(swa_bits, DEV), wst,
                                   wln, cfg.W, cfg.softmax_scale, ws=ws)
        return csa2.csa2_read_device_status(ws)

    big_ok, too_big = np.uint16(0x477F), np.uint16(0x4780)   # 65280 and 65536 as bf16
    assert run(L.q, L.swa) == (0, 0)
    q = L.q.copy(); q[0, 0, 3, 100] = big_ok
    s = L.swa.copy(); s[0, int(inp.win_start[0]), 7] = big_ok | np.uint16(0x8000)
    assert run(q, s) == (0, 0)
    q = L.q.copy(); q[0, 0, 15, 575] = too_big
    st, flags = run(q, L.swa)
    assert st == 6 and flags == csa2.DEV_RANGE
    s = L.swa.copy(); s[0, int(inp.win_start[0]) + int(inp.win_len[0]) - 1, 0] = too_big | np.uint16(0x8000)
    st, flags = run(L.q, s)
    assert st == 6 and flags == csa2.DEV_RANGE
    # a row past the window is not part of the call's input
    end = int(inp.win_start[0]) + int(inp.win_len[0]) - 1
    wl = torch.tensor([int(inp.win_len[0]) - 1], dtype=torch.int32, device=DEV)
    s = L.swa.copy(); s[0, end, 0] = too_big
    csa2.csa2_decode_attention(to_dev_bf16(L.q, DEV), codes, scales, idx, to_dev_bf16(s, DEV), wst, wl, cfg.W,
                               cfg.softmax_scale, ws=ws)
    assert csa2.csa2_read_device_status(ws) == (0, 0)


@pytest.mark.parametrize("B,T,K", [(32, 1, 1024), (64, 1, 1024), (16, 2, 1024), (12, 1, 1024), (4, 1, 2048),
                                   (3, 1, 1900)])
def test_split_merge_through_l2_and_dsmem_agree(B, T, K):
    """With few queries each query's keys are split over a cluster of CTAs: 4 (32 queries),
    2 (64), 8 (12 queries, 9 key tiles) or 16 (4 or 3 queries, 17 or 16 key tiles; the
    last with a ragged split and a window-only split). With a full workspace the partial
    outputs of 2 or 4 splits meet in the exchange at its end (L2), those of 8 or 16 in
    distributed shared memory; with only the status header all meet in distributed shared
    memory. Both must give the oracle's result, and the same result up to summation order."""
    cfg = ci.scaled(ci.DECODE_128K, B=B, N=3000, H=64, K=K, W=128, modes=(ci.FULL,))
    rng = np.random.default_rng(77 + B + T)
    X = rng.standard_normal((B, cfg.N, 576), dtype=np.float32)
    codes, scales = _cache(X)
    q_bits = ci.bf16_bits(rng.standard_normal((B, T, 64, 576), dtype=np.float32) * 0.3)
    swa_bits = ci.bf16_bits(rng.standard_normal((B, 256, 576), dtype=np.float32))
    idx = np.stack([rng.permutation(cfg.N)[:cfg.K] for _ in range(B * T)]).astype(np.int32).reshape(B, T, cfg.K)
    idx[B // 2, 0, 700:] = -1                      # a shorter selection
    wst = np.full(B * T, 100, np.int32)
    wln = np.full(B * T, 128, np.int32)
    wln[1] = 0                                     # an empty window
    q, swa = to_dev_bf16(q_bits, DEV), to_dev_bf16(swa_bits, DEV)
    args = (q, codes, scales, to_dev(idx, DEV), swa, to_dev(wst, DEV), to_dev(wln, DEV), 128, cfg.softmax_scale)
    full_ws = csa2.csa2_workspace(B, T, 64, 0, cfg.K, device=DEV)
    n_sm = torch.cuda.get_device_properties(DEV).multi_processor_count
    nsplit = 1 << int(np.log2(min(16, n_sm // (B * T), (cfg.K + 127) // 128 + 1)))
    assert nsplit == {(32, 1): 4, (64, 1): 2, (16, 2): 4, (12, 1): 8, (4, 1): 16, (3, 1): 16}[B, T]
    if nsplit <= 4:
        assert full_ws.numel() >= 256 + B * T * nsplit * 512 * 64 * 4
    o1, l1 = csa2.csa2_decode_attention(*args, ws=full_ws)
    o2, l2 = csa2.csa2_decode_attention(*args, ws=csa2.csa2_workspace(0, 0, 0, 0, 0, device=DEV))
    torch.cuda.synchronize()
    torch.testing.assert_close(o1, o2, rtol=1e-5, atol=1e-6)
    torch.testing.assert_close(l1, l2, rtol=1e-6, atol=1e-6)
    o1, l1 = o1.cpu().numpy(), l1.cpu().numpy()
    for b in (0, 1, B // 2, B - 1):
        rows = fp4.decode(*fp4.encode(X[b]))
        for t in range(T):
            qi = b * T + t
            sel = idx[b, t][idx[b, t] >= 0]
            O, LSE = attention.attend(f64(q_bits[b, t]), rows[sel], 512, cfg.softmax_scale)
            if wln[qi] > 0:
                Os, Ls = attention.swa_branch(f64(q_bits[b, t]), f64(swa_bits[b]), int(wst[qi]), int(wln[qi]), 512,
                                              cfg.softmax_scale)
                O, LSE = attention.merge(O, LSE, Os, Ls)
            check_attention(o1[b, t], O, f"b={b} t={t}")
            check_lse(l1[b, t], LSE, f"b={b} t={t}")


def test_separate_code_and_scale_rows_equal_the_record_layout():
    """The library's cache keeps an entry's codes and scales in one 384-byte record
    (csa2_kv_cache); code and scale arrays of their own with the same row stride must
    give the same selection prefetch and attention results, bit for bit."""
    cfg = ci.scaled(ci.DECODE_128K, B=4, N=2000, H=64, K=512, W=64, modes=(ci.FULL,))
    inp = ci.make_decode_inputs(cfg)
    L = inp.layers[0]
    codes, scales = _cache(L.X)
    assert scales.data_ptr() == codes.data_ptr() + 288 and codes.stride(-2) == 384
    B, N = codes.shape[:2]
    # separate arrays, same 384-byte row stride, the scales first in their rows
    c2, _ = csa2.csa2_kv_cache((B, N), device=DEV)
    s_buf = torch.full((B, N, 384), 0xEE, dtype=torch.uint8, device=DEV)
    s2 = s_buf[..., :36]
    c2.copy_(codes)
    s2.copy_(scales)
    q = to_dev_bf16(L.q, DEV)
    swa = to_dev_bf16(L.swa, DEV)
    args = dict(q_idx=to_dev_bf16(L.q_idx, DEV), w_idx=to_dev(L.w_idx, DEV), z=to_dev_bf16(L.z, DEV),
                n_visible=to_dev(inp.n_visible, DEV))
    wst, wln = to_dev(inp.win_start, DEV), to_dev(inp.win_len, DEV)
    o1, l1, i1 = csa2.decode_layer(csa2.FULL, q, codes, scales, swa, wst, wln, cfg.W, cfg.K, fused=True, **args)
    o2, l2, i2 = csa2.decode_layer(csa2.FULL, q, c2, s2, swa, wst, wln, cfg.W, cfg.K, fused=True, **args)
    torch.cuda.synchronize()
    assert torch.equal(i1, i2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # a contiguous [B, N, 288] array is not a cache of 384-byte rows
    with pytest.raises(ValueError):
        csa2.csa2_decode_attention(q, codes.contiguous(), scales, i1, swa, wst, wln, cfg.W, cfg.softmax_scale)
