"""Decode-time cache append on the GPU against the oracle: every byte the call writes
(window ring rows, FP4 codes and scales, indexer keys, n_visible, window bounds,
n_tokens) equals the oracle's, and the attention over the appended cache equals the
oracle's attention over the token history.

Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression": blog repost
(sliding window over the most recent n_win tokens), wesearch.press card (4:1 block
compression), picx.dev summary, Methodology / 5 (FP4 entries).
"""
import math

import numpy as np
import pytest
import torch

import csa2_inputs as ci
import sparse_attention_kv_decode_b300 as csa2
from oracle import append as oappend
from oracle import attention, fp4
from tests._util import check_attention, check_lse, f64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rand_state(rng, B, N, S):
    return dict(swa_kv=rng.integers(0, 1 << 16, (B, S, 576), dtype=np.uint16),
                kv_codes=rng.integers(0, 256, (B, N, 288), dtype=np.uint8),
                kv_scales=rng.integers(0, 256, (B, N, 36), dtype=np.uint8),
                z=rng.integers(0, 1 << 16, (B, N, 64), dtype=np.uint16),
                n_visible=rng.integers(-9, 9, B).astype(np.int32),
                win_start=rng.integers(-9, 9, B).astype(np.int32),
                win_len=rng.integers(-9, 9, B).astype(np.int32))


def _dev_state(st):
    d = {}
    for k, v in st.items():
        if v.dtype == np.uint16:
            d[k] = to_dev_bf16(v, DEV)
        elif k not in ("kv_codes", "kv_scales"):
            d[k] = to_dev(v, DEV)
    # the FP4 cache: one 384-byte record per entry
    d["kv_codes"], d["kv_scales"] = csa2.csa2_kv_cache(st["kv_codes"].shape[:2], device=DEV)
    d["kv_codes"].copy_(torch.from_numpy(st["kv_codes"]))
    d["kv_scales"].copy_(torch.from_numpy(st["kv_scales"]))
    return d


def _host(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


@pytest.mark.parametrize("entry_dtype", ["f32", "bf16"])
def test_append_steps_equal_the_oracle_byte_for_byte(entry_dtype):
    rng = np.random.default_rng(41 if entry_dtype == "f32" else 42)
    B, N, n_win, steps = 7, 300, 128, 9
    S = 2 * n_win + 3
    st = _rand_state(rng, B, N, S)
    n_tok = np.array([0, 3, 7, -1, 1001, 126, 131], np.int32)
    dv = _dev_state(st)
    dn = to_dev(n_tok, DEV)
    ws = csa2.csa2_workspace(B, 1, 1, 0, 1, device=DEV)
    for step in range(steps):
        row = ci.bf16_bits(rng.standard_normal((B, 576), dtype=np.float32))
        ent = rng.standard_normal((B, 576), dtype=np.float32) * np.float32(rng.uniform(0.01, 50))
        if entry_dtype == "bf16":
            ent_bits = ci.bf16_bits(ent)
            ent = ci.bf16_bits_to_f32(ent_bits)
            ent_dev = to_dev_bf16(ent_bits, DEV)
        else:
            ent_dev = to_dev(ent, DEV)
        zk = ci.bf16_bits(rng.standard_normal((B, 64), dtype=np.float32))
        csa2.csa2_cache_append(dn, swa_row=to_dev_bf16(row, DEV), swa_kv=dv["swa_kv"], n_win=n_win,
                               entry_kv=ent_dev, entry_z=to_dev_bf16(zk, DEV), kv_codes=dv["kv_codes"],
                               kv_scales=dv["kv_scales"], z=dv["z"], n_visible=dv["n_visible"],
                               win_start=dv["win_start"], win_len=dv["win_len"], ws=ws)
        oappend.cache_append(n_tok, row, st["swa_kv"], n_win, ent, zk, st["kv_codes"], st["kv_scales"], st["z"],
                             st["n_visible"], st["win_start"], st["win_len"])
    torch.cuda.synchronize()
    assert np.array_equal(_host(dn), n_tok)
    for k in st:
        assert np.array_equal(_host(dv[k]), st[k]), k
    assert csa2.csa2_read_device_status(ws) == (0, 0)


def test_entry_past_the_cache_is_flagged_and_skipped():
    rng = np.random.default_rng(43)
    B, N, n_win = 2, 8, 4
    st = _rand_state(rng, B, N, 2 * n_win)
    dv = _dev_state(st)
    dn = to_dev(np.array([4 * N - 1, 4 * N + 3], np.int32), DEV)   # completes entries N-1 and N
    ws = csa2.csa2_workspace(B, 1, 1, 0, 1, device=DEV)
    ent = to_dev(rng.standard_normal((B, 576), dtype=np.float32), DEV)
    csa2.csa2_cache_append(dn, entry_kv=ent, kv_codes=dv["kv_codes"], kv_scales=dv["kv_scales"],
                           n_visible=dv["n_visible"], ws=ws)
    st_code, flags = csa2.csa2_read_device_status(ws)
    assert flags & csa2.DEV_BAD_INDEX
    codes = _host(dv["kv_codes"])
    c, _ = fp4.encode(_host(ent)[0][None, :])
    assert np.array_equal(codes[0, N - 1], c[0])         # last row of the cache written
    assert np.array_equal(codes[1], st["kv_codes"][1])   # nothing written for the entry past it
    assert list(_host(dv["n_visible"])) == [N, N + 1]
    assert list(_host(dn)) == [4 * N, 4 * N + 4]


def test_decode_after_appends_attends_over_the_token_history():
    """Tokens appended one by one from an empty cache; then csa2_decode_attention with
    the appended window bounds and every visible entry selected equals one softmax over
    the FP4 entries (dequantised) and the last n_win token rows of the history."""
    rng = np.random.default_rng(44)
    B, H, n_win, N = 3, 16, 32, 64
    P = [5, 77, 200]                    # tokens per sequence (the window wraps for the last two)
    S = 2 * n_win
    swa = torch.zeros((B, S, 576), dtype=torch.bfloat16, device=DEV)
    codes, scales = csa2.csa2_kv_cache((B, N), device=DEV)
    nvis = torch.zeros(B, dtype=torch.int32, device=DEV)
    wst = torch.zeros(B, dtype=torch.int32, device=DEV)
    wln = torch.zeros(B, dtype=torch.int32, device=DEV)
    n_tok = torch.zeros(B, dtype=torch.int32, device=DEV)
    ws = csa2.csa2_workspace(B, 1, H, N, 64, device=DEV)
    hist_rows = [[] for _ in range(B)]
    hist_ent = [[] for _ in range(B)]
    for p in range(max(P)):
        active = np.array([p < P[b] for b in range(B)])
        nt = torch.where(torch.from_numpy(active).to(DEV), n_tok, torch.full_like(n_tok, -1))
        row = ci.bf16_bits(rng.standard_normal((B, 576), dtype=np.float32))
        ent = rng.standard_normal((B, 576), dtype=np.float32)
        csa2.csa2_cache_append(nt, swa_row=to_dev_bf16(row, DEV), swa_kv=swa, n_win=n_win,
                               entry_kv=to_dev(ent, DEV), kv_codes=codes, kv_scales=scales, n_visible=nvis,
                               win_start=wst, win_len=wln, ws=ws)
        n_tok = torch.where(torch.from_numpy(active).to(DEV), nt, n_tok)
        for b in range(B):
            if active[b]:
                hist_rows[b].append(row[b])
                if (p + 1) % 4 == 0:
                    hist_ent[b].append(ent[b])
    K = N
    nv = _host(nvis)
    idx = np.full((B, 1, K), -1, np.int32)
    for b in range(B):
        idx[b, 0, :nv[b]] = np.arange(nv[b])
    q = ci.bf16_bits(rng.standard_normal((B, 1, H, 576), dtype=np.float32))
    tau = 1.0 / math.sqrt(576)
    o, lse = csa2.csa2_decode_attention(to_dev_bf16(q, DEV), codes, scales, to_dev(idx, DEV), swa, wst, wln,
                                        n_win, softmax_scale=tau, ws=ws)
    torch.cuda.synchronize()
    o, lse = o.cpu().numpy(), lse.cpu().numpy()
    for b in range(B):
        assert nv[b] == P[b] // 4
        ents = np.array(hist_ent[b], np.float32).reshape(-1, 576)
        c, s = fp4.encode(ents)
        keys = np.concatenate([fp4.decode(c, s), f64(np.array(hist_rows[b][-n_win:]))])
        Ow, lw = attention.attend(f64(q[b, 0]), keys, 512, tau)
        check_attention(o[b, 0], Ow, f"sequence {b}")
        check_lse(lse[b, 0], lw, f"sequence {b}")


def test_serving_loop_in_a_cuda_graph():
    """One decode step captured once and replayed per token: csa2_cache_append (advancing
    n_tokens on the device) then csa2_decode_layer(FULL) with the n_visible and window
    bounds the append wrote. K covers every entry, so each token's output is one softmax
    over all entries completed so far and its last n_win tokens."""
    rng = np.random.default_rng(45)
    B, H, H_I, n_win, N, steps = 2, 16, 8, 16, 16, 40
    K = N
    tau = 1.0 / math.sqrt(576)
    dev = DEV
    swa = torch.zeros((B, 2 * n_win, 576), dtype=torch.bfloat16, device=dev)
    codes, scales = csa2.csa2_kv_cache((B, N), device=dev)
    z = torch.zeros((B, N, 64), dtype=torch.bfloat16, device=dev)
    nvis, wst, wln = (torch.zeros(B, dtype=torch.int32, device=dev) for _ in range(3))
    n_tok = torch.tensor([0, 9], dtype=torch.int32, device=dev)     # sequence 1 starts 9 tokens in
    # static per-step inputs, refilled before each replay
    row_in = torch.zeros((B, 576), dtype=torch.bfloat16, device=dev)
    ent_in = torch.zeros((B, 576), dtype=torch.float32, device=dev)
    key_in = torch.zeros((B, 64), dtype=torch.bfloat16, device=dev)
    q_in = torch.zeros((B, 1, H, 576), dtype=torch.bfloat16, device=dev)
    qi_in = torch.zeros((B, 1, H_I, 64), dtype=torch.bfloat16, device=dev)
    w_in = torch.ones((B, 1, H_I), dtype=torch.float32, device=dev)
    idx = torch.empty((B, 1, K), dtype=torch.int32, device=dev)
    o = torch.empty((B, 1, H, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((B, 1, H), dtype=torch.float32, device=dev)
    ws = csa2.csa2_workspace(B, 1, H, N, K, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        csa2.csa2_cache_append(n_tok, swa_row=row_in, swa_kv=swa, n_win=n_win, entry_kv=ent_in, entry_z=key_in,
                               kv_codes=codes, kv_scales=scales, z=z, n_visible=nvis, win_start=wst, win_len=wln,
                               ws=ws, stream=stream)
        csa2.csa2_decode_layer(csa2.FULL, q_in, codes, scales, swa, wst, wln, n_win, K, q_idx=qi_in, w_idx=w_in,
                               z=z, n_visible=nvis, out_idx=idx, o=o, lse=lse, softmax_scale=tau, ws=ws,
                               stream=stream)

    hist_rows, hist_ent = [[], []], [[], []]
    # sequence 1's first 9 tokens: its history before the loop (written by plain appends)
    with torch.cuda.stream(stream):
        pre = torch.tensor([-1, 0], dtype=torch.int32, device=dev)
        for _ in range(9):
            r = ci.bf16_bits(rng.standard_normal((B, 576), dtype=np.float32))
            e = rng.standard_normal((B, 576), dtype=np.float32)
            csa2.csa2_cache_append(pre, swa_row=to_dev_bf16(r, dev), swa_kv=swa, n_win=n_win, entry_kv=to_dev(e, dev),
                                   kv_codes=codes, kv_scales=scales, ws=ws, stream=stream)
            hist_rows[1].append(r[1])
            if len(hist_rows[1]) % 4 == 0:
                hist_ent[1].append(e[1])
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        step()                                   # warm (sets kernel attributes)
    stream.synchronize()
    # the warm step consumed one token per sequence: restart from the same state
    with torch.cuda.stream(stream):
        n_tok.copy_(torch.tensor([0, 9], dtype=torch.int32, device=dev))
    stream.synchronize()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for t in range(steps):
        r = ci.bf16_bits(rng.standard_normal((B, 576), dtype=np.float32))
        e = rng.standard_normal((B, 576), dtype=np.float32)
        q = ci.bf16_bits(rng.standard_normal((B, 1, H, 576), dtype=np.float32))
        with torch.cuda.stream(stream):   # inputs and replay on the graph's stream, in order
            row_in.copy_(to_dev_bf16(r, dev))
            ent_in.copy_(to_dev(e, dev))
            q_in.copy_(to_dev_bf16(q, dev))
            graph.replay()
        stream.synchronize()
        for b in range(B):
            hist_rows[b].append(r[b])
            if len(hist_rows[b]) % 4 == 0:
                hist_ent[b].append(e[b])
            keys = [f64(np.array(hist_rows[b][-n_win:]))]
            if hist_ent[b]:
                c, s = fp4.encode(np.array(hist_ent[b], np.float32))
                keys.insert(0, fp4.decode(c, s))
            Ow, lw = attention.attend(f64(q[b, 0]), np.concatenate(keys), 512, tau)
            check_attention(o[b, 0].cpu().numpy(), Ow, f"token {t} sequence {b}")
            check_lse(lse[b, 0].cpu().numpy(), lw, f"token {t} sequence {b}")
    assert _host(n_tok).tolist() == [steps, 9 + steps]
    assert csa2.csa2_read_device_status(ws) == (0, 0)
