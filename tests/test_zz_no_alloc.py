"""csa2_index_topk_noalloc: csa2_index_topk on the library's fixed device scratch.

The call allocates nothing and takes no workspace, for callers that cannot allocate
device memory (an engine that has reserved all of it for its own KV pool, a plug-in
given tensors but no allocator). It must return what the workspace call returns for
the same inputs, call after call (the scratch keeps whatever the previous call left in
it). The file is collected last, and it also passes when run alone in a fresh process
(then its first call does the per-device set-up).

Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", picx.dev summary,
Methodology / 2. CSA2 (the indexer's top-K of FULL / REINDEX, and REUSE).
"""

import numpy as np
import pytest
import torch

import csa2_inputs as ci
import sparse_attention_kv_decode_b300 as csa2
from tests._util import to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _layer(cfg):
    inp = ci.make_decode_inputs(cfg, with_x=False)
    L = inp.layers[0]
    return (to_dev_bf16(L.q_idx, "cuda"), to_dev(L.w_idx, "cuda"), to_dev_bf16(L.z, "cuda"),
            to_dev(inp.n_visible.astype(np.int32), "cuda"))


def _same(a, b):
    assert torch.equal(a, b)


@pytest.mark.parametrize("B,N,K,H_I", [(3, 5000, 512, 8), (32, 32768, 2048, 8)])
def test_matches_workspace_call_twice(B, N, K, H_I):
    cfg = ci.scaled(ci.DECODE_128K, B=B, N=N, H=16, H_I=H_I, K=K, W=8, modes=(ci.FULL,))
    q, w, z, nv = _layer(cfg)
    want_s = torch.empty((B, 1, K), dtype=torch.float32, device="cuda")
    want = csa2.csa2_index_topk(csa2.FULL, q, w, z, nv, K, out_scores=want_s)
    torch.cuda.synchronize()
    for mode in (csa2.FULL, csa2.REINDEX):
        for _ in range(2):
            got = torch.full((B, 1, K), -7, dtype=torch.int32, device="cuda")
            got_s = torch.empty((B, 1, K), dtype=torch.float32, device="cuda")
            csa2.csa2_index_topk_noalloc(mode, q, w, z, nv, K, got, out_scores=got_s)
            torch.cuda.synchronize()
            _same(got, want)
            _same(got_s.view(torch.int32), want_s.view(torch.int32))


def test_reuse_copies_prev():
    prev = torch.arange(2 * 3 * 64, dtype=torch.int32, device="cuda").reshape(2, 3, 64)
    out = torch.full_like(prev, -7)
    csa2.csa2_index_topk_noalloc(csa2.REUSE, None, None, None, None, 64, out, prev_idx=prev)
    torch.cuda.synchronize()
    _same(out, prev)


def test_rejects_more_scores_than_the_scratch_holds():
    # 32 queries x 66,560 padded entries > 2^21 scores: refused before any launch
    B, N, K, H_I = 32, 65537, 2048, 8
    q = torch.zeros((B, 1, H_I, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.ones((B, 1, H_I), dtype=torch.float32, device="cuda")
    z = torch.zeros((B, N, 64), dtype=torch.bfloat16, device="cuda")
    nv = torch.full((B,), N, dtype=torch.int32, device="cuda")
    out = torch.full((B, 1, K), -7, dtype=torch.int32, device="cuda")
    L = csa2.lib()
    st = L.csa2_index_topk_noalloc(csa2.FULL, B, 1, H_I, q.data_ptr(), w.data_ptr(), z.data_ptr(), N,
                                   nv.data_ptr(), K, None, out.data_ptr(), None, None)
    assert st == 3  # CSA2_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == -7).all())
    # one entry fewer per query still fits: 32 x 65,536 = 2^21
    nv2 = torch.full((B,), 65536, dtype=torch.int32, device="cuda")
    st = L.csa2_index_topk_noalloc(csa2.FULL, B, 1, H_I, q.data_ptr(), w.data_ptr(), z.data_ptr(), 65536,
                                   nv2.data_ptr(), K, None, out.data_ptr(), None, None)
    assert st == 0
    torch.cuda.synchronize()
    # all scores are 0: the K lowest indices win the ties
    assert bool((out == torch.arange(K, dtype=torch.int32, device="cuda")).all())


def test_leftover_scores_under_the_range_words_of_a_larger_call():
    """The per-query range words sit after the header and the scores after them, both
    placed by the call's own query count: a 32-query call leaves scores where a later
    64-query call keeps its range words. The selection must stay exact from that start."""
    N, K = 32768, 2048
    for B in (32, 64, 32):
        cfg = ci.scaled(ci.DECODE_128K, B=B, N=N, H=16, K=K, W=8, modes=(ci.FULL,), seed=B)
        q, w, z, nv = _layer(cfg)
        want_s = torch.empty((B, 1, K), dtype=torch.float32, device="cuda")
        want = csa2.csa2_index_topk(csa2.FULL, q, w, z, nv, K, out_scores=want_s)
        got = torch.full((B, 1, K), -7, dtype=torch.int32, device="cuda")
        got_s = torch.empty((B, 1, K), dtype=torch.float32, device="cuda")
        csa2.csa2_index_topk_noalloc(csa2.FULL, q, w, z, nv, K, got, out_scores=got_s)
        torch.cuda.synchronize()
        _same(got, want)
        _same(got_s.view(torch.int32), want_s.view(torch.int32))


def test_reindex_pool_matches_workspace_call():
    """REINDEX_POOL through the fixed scratch: its score rows are pool-sized, so 32 queries
    with K = 2048 fit at any cache length (here 100,000 entries, where a full scan would not
    fit). Compared bit for bit with the workspace call, twice in a row."""
    B, N, K, H_I = 32, 100000, 2048, 8
    g = torch.Generator(device="cuda").manual_seed(12)
    q = torch.randn((B, 1, H_I, 64), generator=g, device="cuda").to(torch.bfloat16)
    w = torch.randn((B, 1, H_I), generator=g, device="cuda").abs()
    z = torch.randn((B, N, 64), generator=g, device="cuda").to(torch.bfloat16)
    nv = torch.randint(N // 2, N + 1, (B,), generator=g, device="cuda", dtype=torch.int32)
    full_sel = csa2.csa2_index_topk(csa2.FULL, q, w, z, nv, K)
    q2 = torch.randn((B, 1, H_I, 64), generator=g, device="cuda").to(torch.bfloat16)
    z2 = torch.randn((B, N, 64), generator=g, device="cuda").to(torch.bfloat16)
    want_s = torch.empty((B, 1, K), dtype=torch.float32, device="cuda")
    want = csa2.csa2_index_topk(csa2.REINDEX_POOL, q2, w, z2, nv, K, prev_idx=full_sel, out_scores=want_s)
    torch.cuda.synchronize()
    for _ in range(2):
        got = torch.full((B, 1, K), -7, dtype=torch.int32, device="cuda")
        got_s = torch.empty((B, 1, K), dtype=torch.float32, device="cuda")
        csa2.csa2_index_topk_noalloc(csa2.REINDEX_POOL, q2, w, z2, nv, K, got, prev_idx=full_sel,
                                     out_scores=got_s)
        torch.cuda.synchronize()
        _same(got, want)
        _same(got_s.view(torch.int32), want_s.view(torch.int32))
    # the full scan of the same call does not fit the scratch and is refused
    with pytest.raises(csa2.Csa2Error) as ex:
        csa2.csa2_index_topk_noalloc(csa2.REINDEX, q2, w, z2, nv, K, got)
    assert ex.value.status == 3
