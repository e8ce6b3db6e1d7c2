"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, and rejects bad arguments before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa2.h")


@pytest.fixture(scope="module")
def L():
    from sparse_attention_kv_decode_b300 import _build
    _build.build()
    import sparse_attention_kv_decode_b300 as csa2
    return csa2.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"CSA2_API\s+[\w\s\*]*?\b(csa2_\w+)\s*\(", text)))


def test_header_declares_the_four_path_calls():
    names = declared_symbols()
    for n in ("csa2_encode_kv", "csa2_index_topk", "csa2_sparse_decode", "csa2_swa_merge"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name


def test_version_and_status_strings(L):
    assert L.csa2_version() == 200
    for s in range(7):
        assert L.csa2_status_string(s)
    assert L.csa2_status_string(99) == b"unknown status"


FAKE = 0x10000  # aligned, never dereferenced: every call below fails validation first


def test_index_topk_validation(L):
    r = L.csa2_index_topk
    assert r(7, 1, 1, 4, FAKE, FAKE, FAKE, 1024, FAKE, 128, None, FAKE, None, FAKE, 1 << 30, None) == 1
    assert r(0, 1, 1, 4, FAKE, FAKE, FAKE, 1024, FAKE, 5000, None, FAKE, None, FAKE, 1 << 30, None) == 2
    assert r(0, 1, 1, 17, FAKE, FAKE, FAKE, 1024, FAKE, 128, None, FAKE, None, FAKE, 1 << 30, None) == 2
    assert r(0, 1, 1, 4, FAKE, FAKE, FAKE, 1 << 21, FAKE, 128, None, FAKE, None, FAKE, 1 << 30, None) == 2
    assert r(0, 1, 1, 4, None, FAKE, FAKE, 1024, FAKE, 128, None, FAKE, None, FAKE, 1 << 30, None) == 1
    assert r(0, 1, 1, 4, FAKE + 2, FAKE, FAKE, 1024, FAKE, 128, None, FAKE, None, FAKE, 1 << 30, None) == 1
    assert r(0, 1, 1, 4, FAKE, FAKE, FAKE, 1024, FAKE, 128, None, FAKE, None, None, 0, None) == 3
    assert r(0, 1, 1, 4, FAKE, FAKE, FAKE, 1024, FAKE, 128, None, FAKE, None, FAKE, 1024, None) == 3
    assert r(0, 1, 1, 4, FAKE, FAKE, FAKE, 1024, FAKE, 128, None, FAKE, None, FAKE + 16, 1 << 30, None) == 1
    # REUSE needs the preceding layer's indices
    assert r(2, 1, 1, 0, None, None, None, 0, None, 128, None, FAKE, None, None, 0, None) == 1
    # REUSE with out == prev is a no-op that launches nothing
    assert r(2, 1, 1, 0, None, None, None, 0, None, 128, FAKE, FAKE, None, None, 0, None) == 0


def test_sparse_decode_validation(L):
    r = L.csa2_sparse_decode
    ok = dict()
    assert r(1, 1, 20, FAKE, FAKE, FAKE, 1024, FAKE, 128, 512, ctypes.c_float(0.04), FAKE, FAKE, FAKE, 1 << 30, None) == 2
    assert r(1, 1, 64, FAKE, FAKE, FAKE, 1024, FAKE, 128, 576, ctypes.c_float(0.04), FAKE, FAKE, FAKE, 1 << 30, None) == 2
    assert r(1, 1, 64, FAKE, FAKE, FAKE, 1024, FAKE, 8192, 512, ctypes.c_float(0.04), FAKE, FAKE, FAKE, 1 << 30, None) == 2
    assert r(1, 1, 64, None, FAKE, FAKE, 1024, FAKE, 128, 512, ctypes.c_float(0.04), FAKE, FAKE, FAKE, 1 << 30, None) == 1
    assert r(1, 1, 64, FAKE, FAKE + 8, FAKE, 1024, FAKE, 128, 512, ctypes.c_float(0.04), FAKE, FAKE, FAKE, 1 << 30, None) == 1
    assert r(1, 1, 64, FAKE, FAKE, FAKE, 1024, FAKE, 128, 512, ctypes.c_float(float("nan")), FAKE, FAKE, FAKE, 1 << 30, None) == 1
    assert r(1, 1, 64, FAKE, FAKE, FAKE, 1024, FAKE, 128, 512, ctypes.c_float(0.04), FAKE, FAKE, None, 0, None) == 3
    assert r(1, 1, 64, FAKE, FAKE, FAKE, 1024, FAKE, 128, 512, ctypes.c_float(0.04), FAKE, FAKE, FAKE, 128, None) == 3
    # empty batch: nothing to do
    assert r(0, 1, 64, None, None, None, 0, None, 128, 512, ctypes.c_float(0.04), None, None, None, 0, None) == 0


def test_swa_merge_validation(L):
    r = L.csa2_swa_merge
    f = ctypes.c_float(0.04)
    assert r(1, 1, 64, FAKE, FAKE, 128, FAKE, FAKE, 300, 512, f, FAKE, FAKE, FAKE, None, FAKE, 1 << 30, None) == 2
    assert r(1, 1, 64, FAKE, FAKE, 128, FAKE, FAKE, 128, 512, f, None, FAKE, FAKE, None, FAKE, 1 << 30, None) == 1
    assert r(1, 1, 64, FAKE, FAKE, 128, FAKE, FAKE, 128, 512, f, FAKE, FAKE, FAKE, None, None, 0, None) == 3
    assert r(1, 1, 64, FAKE, FAKE, -1, FAKE, FAKE, 128, 512, f, FAKE, FAKE, FAKE, None, FAKE, 1 << 30, None) == 1


def test_encode_validation(L):
    r = L.csa2_encode_kv
    # quantise-only needs d_model == 576 and n_layers == 1
    assert r(FAKE, 0, 16, 512, None, None, 1, FAKE, FAKE, None, None, 0, None) == 1
    assert r(FAKE, 0, 16, 576, None, None, 2, FAKE, FAKE, None, None, 0, None) == 1
    assert r(FAKE, 5, 16, 576, None, None, 1, FAKE, FAKE, None, None, 0, None) == 1
    assert r(FAKE + 4, 0, 16, 576, None, None, 1, FAKE, FAKE, None, None, 0, None) == 1
    # projection: bf16 only, d_model multiple of 64, all outputs present
    assert r(FAKE, 0, 16, 4096, FAKE, FAKE, 20, FAKE, FAKE, FAKE, None, 0, None) == 1
    assert r(FAKE, 1, 16, 4000, FAKE, FAKE, 20, FAKE, FAKE, FAKE, None, 0, None) == 1
    assert r(FAKE, 1, 16, 4096, FAKE, FAKE, 20, FAKE, FAKE, None, None, 0, None) == 1
    assert r(FAKE, 1, 0, 4096, FAKE, FAKE, 20, FAKE, FAKE, FAKE, None, 0, None) == 0
    # projection needs the workspace status word
    assert r(FAKE, 1, 16, 4096, FAKE, FAKE, 20, FAKE, FAKE, FAKE, None, 0, None) == 3
    assert r(FAKE, 1, 16, 4096, FAKE, FAKE, 20, FAKE, FAKE, FAKE, FAKE, 128, None) == 3


def test_workspace_size_monotone(L):
    a = L.csa2_workspace_bytes(32, 1, 64, 32768, 2048)
    b = L.csa2_workspace_bytes(32, 1, 64, 65536, 2048)
    c = L.csa2_workspace_bytes(64, 1, 64, 65536, 2048)
    assert 256 < a <= b <= c
    # header + range words + fp32 scores + the candidate pool of a REINDEX call (block ids
    # [Q][K] and one visible count per query) + the attention's split exchange (up to 4
    # splits x 512 dims x 64 heads fp32 per query, for at most 128 queries)
    xchg = 4 * 512 * 64 * 4
    assert a == 256 + 256 + 32 * 32768 * 4 + 32 * 2048 * 4 + 256 + 32 * xchg
    assert L.csa2_workspace_bytes(1, 1, 64, 0, 2048) == 512 + 2048 * 4 + 256 + xchg
    assert L.csa2_workspace_bytes(129, 1, 64, 0, 1) == 256 + 1280 + 768 + 768   # no exchange past 128
    assert L.csa2_workspace_bytes(-1, 1, 64, 10, 10) == 0


def test_decode_attention_validation(L):
    r = L.csa2_decode_attention
    f = ctypes.c_float(0.04)
    args = [1, 1, 64, FAKE, FAKE, FAKE, 1024, FAKE, 128, FAKE, 128, FAKE, FAKE, 128, 512, f, FAKE, FAKE, FAKE,
            1 << 30, None]

    def call(**kw):
        a = list(args)
        for k, v in kw.items():
            a[int(k[1:])] = v
        return r(*a)

    assert call(a2=20) == 2                       # heads not a multiple of 16
    assert call(a13=300) == 2                     # window longer than 256
    assert call(a8=5000) == 2                     # K above 4096
    assert call(a14=576) == 2                     # d_v must be 512
    assert call(a3=None) == 1                     # q missing
    assert call(a9=None) == 1                     # window rows missing with s_stride > 0
    assert call(a3=FAKE + 8) == 1                 # q not 16-byte aligned
    assert call(a15=ctypes.c_float(float("nan"))) == 1
    assert call(a18=None, a19=0) == 3             # no workspace
    assert call(a19=128) == 3                     # workspace below the status header
    assert call(a0=0) == 0                        # empty batch: nothing to do


def test_decode_layer_validation(L):
    """Both halves of csa2_decode_layer are checked before anything launches (no GPU)."""
    r = L.csa2_decode_layer
    f = ctypes.c_float(0.04)
    # mode, B, T, H, H_I, q, q_idx, w_idx, z, codes, scales, N, n_visible, K, prev, out_idx,
    # swa, S, win_start, win_len, n_win, d_v, scale, o, lse, ws, ws_bytes, stream
    args = [0, 1, 1, 64, 8, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1024, FAKE, 128, None, FAKE,
            FAKE, 128, FAKE, FAKE, 128, 512, f, FAKE, FAKE, FAKE, 1 << 30, None]

    def call(**kw):
        a = list(args)
        for k, v in kw.items():
            a[int(k[1:])] = v
        return r(*a)

    assert call(a3=20) == 2                       # attention: heads not a multiple of 16
    assert call(a20=300) == 2                     # attention: window longer than 256
    assert call(a21=576) == 2                     # attention: d_v must be 512
    assert call(a13=5000) == 2                    # K above 4096
    assert call(a4=17) == 2                       # selection: more than 16 indexer heads
    assert call(a0=7) == 1                        # unknown mode
    assert call(a5=None) == 1                     # q missing
    assert call(a6=None) == 1                     # q_idx missing (FULL)
    assert call(a15=None) == 1                    # out_idx missing
    assert call(a0=2, a14=None) == 1              # REUSE without prev_idx
    assert call(a22=ctypes.c_float(float("nan"))) == 1
    assert call(a25=None, a26=0) == 3             # no workspace
    assert call(a26=4096) == 3                    # workspace without room for the scores
    assert call(a1=0) == 0                        # empty batch: nothing to do


def test_cache_append_validation(L):
    """csa2_cache_append rejects bad arguments before launching (no GPU)."""
    r = L.csa2_cache_append
    # B, n_tokens, advance, ratio, swa_row, swa_kv, S, n_win, entry_kv, entry_dtype, entry_z,
    # codes, scales, z, N, n_visible, win_start, win_len, ws, ws_bytes, stream
    args = [4, FAKE, 1, 4, FAKE, FAKE, 256, 128, FAKE, 0, FAKE, FAKE, FAKE, FAKE, 1024, FAKE, FAKE, FAKE,
            FAKE, 1 << 20, None]

    def call(**kw):
        a = list(args)
        for k, v in kw.items():
            a[int(k[1:])] = v
        return r(*a)

    assert call(a3=0) == 1                        # ratio below 1
    assert call(a6=255) == 1                      # ring store shorter than 2 * n_win
    assert call(a7=0) == 1                        # a window row without a window
    assert call(a4=None, a7=0) == 1               # window bounds requested without a window
    assert call(a17=None) == 1                    # win_start without win_len
    assert call(a5=None) == 1                     # window row without a store
    assert call(a4=FAKE + 8) == 1                 # misaligned window row
    assert call(a9=5) == 1                        # unknown entry dtype
    assert call(a11=None) == 1                    # entry without codes
    assert call(a13=None) == 1                    # key without z
    assert call(a1=None) == 1                     # n_tokens missing
    assert call(a18=None, a19=0) == 3             # no workspace (status word)
    assert call(a19=64) == 3                      # workspace smaller than the header
    assert call(a0=0) == 0                        # empty batch: nothing to do
    assert call(a0=0, a1=None) == 0


def test_check_bounded_wait_validation(L):
    r = L.csa2_check_bounded_wait
    assert r(999, FAKE, 1 << 20, None) == 1            # bound below a microsecond
    assert r(2_000_000_000, FAKE, 1 << 20, None) == 1  # above the kernels' own one-second bound
    assert r(1_000_000, None, 0, None) == 3            # no workspace (status word)
    assert r(1_000_000, FAKE, 64, None) == 3           # workspace smaller than the header


def test_binding_declares_argument_types_for_every_entry_point(L):
    """Every call of the header has its C signature declared in the binding (ctypes would
    otherwise pass 64-bit sizes and pointers as C ints)."""
    for name in declared_symbols():
        fn = getattr(L, name)
        if name in ("csa2_version", "csa2_last_cuda_error"):
            continue
        assert fn.argtypes is not None, name
