"""Python binding of libcsa2, the CSA2 FP4 sparse-decode library for B300 (sm_103a).

Argument marshalling only: every step runs in the CUDA kernels of libcsa2.so,
reached through its C ABI (include/csa2.h) with ctypes. Tensors are PyTorch
CUDA tensors (PyTorch provides device memory and streams); bf16 tensors may be
torch.bfloat16 or 16-bit integer views of the same bits. The binding raises
Csa2Error on any non-zero status and RuntimeError when the library is missing;
there is no fallback path.

Functions carry the C names:
  csa2_encode_kv       FP4 quantise-only write, or the CED projection Eq. (1)
  csa2_index_topk      indexer scores + top-K (FULL / REINDEX), or REUSE
  csa2_sparse_decode   sparse MQA over the selected FP4 entries (global branch)
  csa2_swa_merge       sliding-window branch + log-sum-exp merge
plus csa2_workspace / csa2_read_device_status helpers and decode_layer(), which
chains the three decode calls of one CSA2 layer.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libcsa2.so")

FULL, REINDEX, REUSE, REINDEX_POOL = 0, 1, 2, 3
F32, BF16 = 0, 1
D_KV, D_LATENT, D_IDX = 576, 512, 64
CODE_BYTES, SCALE_BYTES, ENTRY_BYTES = 288, 36, 384

STATUS = {0: "CSA2_OK", 1: "CSA2_ERR_INVALID_ARG", 2: "CSA2_ERR_UNSUPPORTED", 3: "CSA2_ERR_WORKSPACE",
          4: "CSA2_ERR_CUDA", 5: "CSA2_ERR_TIMEOUT", 6: "CSA2_ERR_DEVICE_CHECK"}
DEV_BAD_INDEX, DEV_BAD_WINDOW, DEV_TOPK_LEVELS, DEV_PIPELINE_TIMEOUT, DEV_RANGE = 0x1, 0x2, 0x4, 0x8, 0x10

_LIB = None


class Csa2Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {STATUS.get(status, status)} ({_lib().csa2_status_string(status).decode()})"
        if status == 4:
            msg += f": {_lib().csa2_last_cuda_error().decode()}"
        super().__init__(msg)


def _lib():
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libcsa2.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    L.csa2_encode_kv.argtypes = [vp, i32, i64, i32, vp, vp, i32, vp, vp, vp, vp, sz, vp]
    L.csa2_index_topk.argtypes = [i32, i32, i32, i32, vp, vp, vp, i64, vp, i32, vp, vp, vp, vp, sz, vp]
    L.csa2_index_topk_noalloc.argtypes = [i32, i32, i32, i32, vp, vp, vp, i64, vp, i32, vp, vp, vp, vp]
    L.csa2_sparse_decode.argtypes = [i32, i32, i32, vp, vp, vp, i64, vp, i32, i32, f32, vp, vp, vp, sz, vp]
    L.csa2_decode_attention.argtypes = [i32, i32, i32, vp, vp, vp, i64, vp, i32, vp, i64, vp, vp, i32, i32, f32,
                                        vp, vp, vp, sz, vp]
    L.csa2_index_topk_prefetch.argtypes = [i32, i32, i32, i32, vp, vp, vp, i64, vp, i32, vp, vp, vp, vp, vp,
                                           vp, sz, vp]
    L.csa2_decode_layer.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i64, vp, i32, vp, vp,
                                    vp, i64, vp, vp, i32, i32, f32, vp, vp, vp, sz, vp]
    L.csa2_swa_merge.argtypes = [i32, i32, i32, vp, vp, i64, vp, vp, i32, i32, f32, vp, vp, vp, vp, vp, sz, vp]
    L.csa2_cache_append.argtypes = [i32, vp, i32, i32, vp, vp, i64, i32, vp, i32, vp, vp, vp, vp, i64, vp, vp,
                                    vp, vp, sz, vp]
    L.csa2_check_bounded_wait.argtypes = [i64, vp, sz, vp]
    L.csa2_workspace_bytes.argtypes = [i32, i32, i32, i64, i32]
    L.csa2_workspace_bytes.restype = sz
    L.csa2_workspace_init.argtypes = [vp, sz, vp]
    L.csa2_read_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    L.csa2_status_string.argtypes = [i32]
    L.csa2_status_string.restype = ctypes.c_char_p
    L.csa2_version.argtypes = []
    L.csa2_last_cuda_error.argtypes = []
    L.csa2_last_cuda_error.restype = ctypes.c_char_p
    for fn in ("csa2_encode_kv", "csa2_index_topk", "csa2_index_topk_prefetch", "csa2_sparse_decode",
               "csa2_swa_merge", "csa2_decode_layer", "csa2_cache_append", "csa2_check_bounded_wait",
               "csa2_workspace_init", "csa2_read_device_status", "csa2_version"):
        getattr(L, fn).restype = ctypes.c_int
    _LIB = L
    return L


def lib():
    """The loaded ctypes library (raises if it is not built)."""
    return _lib()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != 0:
        raise Csa2Error(status, what)


def _dev(t: torch.Tensor, name: str, dtypes, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")
    return t


def _dev_kv(t: torch.Tensor, name: str, lead, width: int):
    """kv_codes / kv_scales: uint8 [*lead, width] whose rows are ENTRY_BYTES apart."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.uint8:
        raise ValueError(f"{name}: dtype {t.dtype} is not uint8")
    if lead is not None and tuple(t.shape) != tuple(lead) + (width,):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(lead) + (width,)}")
    expect = ENTRY_BYTES
    ok = t.stride(-1) == 1
    for d in range(t.dim() - 2, -1, -1):
        ok = ok and (t.shape[d] == 1 or t.stride(d) == expect)
        expect *= t.shape[d]
    if not ok:
        raise ValueError(f"{name}: rows must be {ENTRY_BYTES} bytes apart (use csa2_kv_cache)")
    return t


def csa2_kv_cache(lead, device=None):
    """A zeroed FP4 cache of entries [*lead]: one ENTRY_BYTES record per entry holding
    the 288 code bytes, the 36 scale bytes and 60 bytes of padding. Returns the
    (codes [*lead, 288], scales [*lead, 36]) views the calls take."""
    kv = torch.zeros(tuple(lead) + (ENTRY_BYTES,), dtype=torch.uint8, device=device)
    return kv[..., :CODE_BYTES], kv[..., CODE_BYTES:CODE_BYTES + SCALE_BYTES]


_B16 = (torch.bfloat16, torch.int16, torch.uint16)


# ---------------------------------------------------------------------------
# Workspace
# ---------------------------------------------------------------------------
def csa2_workspace_bytes(B: int, T: int, H: int, n_max: int, K: int) -> int:
    return int(_lib().csa2_workspace_bytes(B, T, H, n_max, K))


def csa2_workspace(B: int, T: int, H: int, n_max: int, K: int, device=None, stream=None) -> torch.Tensor:
    """Allocate (through PyTorch) and initialise a workspace covering these sizes."""
    nbytes = csa2_workspace_bytes(B, T, H, n_max, K)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
    _check(_lib().csa2_workspace_init(ws.data_ptr(), nbytes, _stream(stream)), "csa2_workspace_init")
    return ws


def csa2_read_device_status(ws: torch.Tensor, stream=None) -> Tuple[int, int]:
    """(status, flags): synchronises the stream and clears the device status word."""
    flags = ctypes.c_uint32(0)
    st = _lib().csa2_read_device_status(ws.data_ptr(), _stream(stream), ctypes.byref(flags))
    return st, flags.value


# ---------------------------------------------------------------------------
# Entry points
# ---------------------------------------------------------------------------
def csa2_encode_kv(h: torch.Tensor, w_kv: Optional[torch.Tensor] = None, w_z: Optional[torch.Tensor] = None,
                   kv_codes: Optional[torch.Tensor] = None, kv_scales: Optional[torch.Tensor] = None,
                   z_out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, stream=None):
    """Quantise rows h [..., 576] (fp32/bf16) to FP4, or run the CED projection.

    Quantise-only returns (codes [..., 288] u8, scales [..., 36] u8), views of one
    record per entry (csa2_kv_cache). With w_kv [L, 576, d] and w_z [L, 64, d] (bf16),
    h is bf16 [rows, d] and the result is (codes [L, rows, 288], scales [L, rows, 36],
    z [L, rows, 64] bf16).
    """
    L = _lib()
    if w_kv is None and w_z is None:
        _dev(h, "h", (torch.float32,) + _B16)
        if h.shape[-1] != D_KV:
            raise ValueError("h must have 576 channels")
        lead = tuple(h.shape[:-1])
        rows = h.numel() // D_KV
        if kv_codes is None and kv_scales is None:
            kv_codes, kv_scales = csa2_kv_cache(lead, device=h.device)
        _dev_kv(kv_codes, "kv_codes", lead, CODE_BYTES)
        _dev_kv(kv_scales, "kv_scales", lead, SCALE_BYTES)
        dt = F32 if h.dtype == torch.float32 else BF16
        _check(L.csa2_encode_kv(_ptr(h), dt, rows, D_KV, None, None, 1, _ptr(kv_codes), _ptr(kv_scales),
                                None, None, 0, _stream(stream)), "csa2_encode_kv")
        return kv_codes, kv_scales
    _dev(h, "h", _B16)
    rows, d_model = h.shape
    n_layers = w_kv.shape[0]
    _dev(w_kv, "w_kv", _B16, (n_layers, D_KV, d_model))
    _dev(w_z, "w_z", _B16, (n_layers, D_IDX, d_model))
    if kv_codes is None and kv_scales is None:
        kv_codes, kv_scales = csa2_kv_cache((n_layers, rows), device=h.device)
    if z_out is None:
        z_out = torch.empty((n_layers, rows, D_IDX), dtype=torch.bfloat16, device=h.device)
    _dev_kv(kv_codes, "kv_codes", (n_layers, rows), CODE_BYTES)
    _dev_kv(kv_scales, "kv_scales", (n_layers, rows), SCALE_BYTES)
    _dev(z_out, "z_out", _B16, (n_layers, rows, D_IDX))
    if ws is None:
        ws = csa2_workspace(0, 0, 0, 0, 0, device=h.device, stream=stream)
    _check(L.csa2_encode_kv(_ptr(h), BF16, rows, d_model, _ptr(w_kv), _ptr(w_z), n_layers, _ptr(kv_codes),
                            _ptr(kv_scales), _ptr(z_out), _ptr(ws), ws.numel(), _stream(stream)), "csa2_encode_kv")
    return kv_codes, kv_scales, z_out


def csa2_index_topk(mode: int, q_idx: Optional[torch.Tensor], w_idx: Optional[torch.Tensor],
                    z: Optional[torch.Tensor], n_visible: Optional[torch.Tensor], K: int,
                    prev_idx: Optional[torch.Tensor] = None, out_idx: Optional[torch.Tensor] = None,
                    out_scores: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                    B: Optional[int] = None, T: Optional[int] = None, stream=None) -> torch.Tensor:
    """Top-K indices [B, T, K] int32 (ascending, -1 padded) of one CSA2 layer.

    FULL/REINDEX: q_idx [B, T, H_I, 64] bf16, w_idx [B, T, H_I] fp32, z [B, N, 64] bf16,
    n_visible [B*T] int32. REUSE: returns prev_idx's values (in out_idx if given).
    """
    L = _lib()
    if mode == REUSE:
        if prev_idx is None:
            raise ValueError("REUSE needs prev_idx")
        _dev(prev_idx, "prev_idx", (torch.int32,))
        B_, T_, K_ = prev_idx.shape
        if out_idx is None:
            return prev_idx
        _dev(out_idx, "out_idx", (torch.int32,), prev_idx.shape)
        _check(L.csa2_index_topk(REUSE, B_, T_, 0, None, None, None, 0, None, K_, _ptr(prev_idx), _ptr(out_idx),
                                 None, None, 0, _stream(stream)), "csa2_index_topk(REUSE)")
        return out_idx
    _dev(q_idx, "q_idx", _B16)
    B_, T_, H_I, _ = q_idx.shape
    _dev(w_idx, "w_idx", (torch.float32,), (B_, T_, H_I))
    _dev(z, "z", _B16)
    N = z.shape[1]
    if z.shape != (B_, N, D_IDX):
        raise ValueError("z must be [B, N, 64]")
    _dev(n_visible, "n_visible", (torch.int32,), (B_ * T_,))
    if mode == REINDEX_POOL:
        if prev_idx is None:
            raise ValueError("REINDEX_POOL needs the FULL layer's selection as prev_idx")
        _dev(prev_idx, "prev_idx", (torch.int32,), (B_, T_, K))
    if out_idx is None:
        out_idx = torch.empty((B_, T_, K), dtype=torch.int32, device=q_idx.device)
    _dev(out_idx, "out_idx", (torch.int32,), (B_, T_, K))
    if out_scores is not None:
        _dev(out_scores, "out_scores", (torch.float32,), (B_, T_, K))
    if ws is None:
        ws = csa2_workspace(B_, T_, 0, N, K, device=q_idx.device, stream=stream)
    _check(L.csa2_index_topk(mode, B_, T_, H_I, _ptr(q_idx), _ptr(w_idx), _ptr(z), N, _ptr(n_visible), K,
                             _ptr(prev_idx), _ptr(out_idx), _ptr(out_scores), _ptr(ws), ws.numel(),
                             _stream(stream)), "csa2_index_topk")
    return out_idx


def csa2_index_topk_noalloc(mode: int, q_idx: Optional[torch.Tensor], w_idx: Optional[torch.Tensor],
                            z: Optional[torch.Tensor], n_visible: Optional[torch.Tensor], K: int,
                            out_idx: torch.Tensor, prev_idx: Optional[torch.Tensor] = None,
                            out_scores: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """csa2_index_topk on the library's fixed device scratch: no workspace, and
    nothing is allocated (out_idx [B, T, K] int32 is the caller's). REUSE and
    REINDEX_POOL take prev_idx [B, T, K] int32 (REINDEX_POOL: the FULL layer's selection)."""
    L = _lib()
    _dev(out_idx, "out_idx", (torch.int32,))
    B_, T_, K_ = out_idx.shape
    if K_ != K:
        raise ValueError("out_idx must be [B, T, K]")
    if mode == REUSE:
        if prev_idx is None:
            raise ValueError("REUSE needs prev_idx")
        _dev(prev_idx, "prev_idx", (torch.int32,), out_idx.shape)
        _check(L.csa2_index_topk_noalloc(REUSE, B_, T_, 0, None, None, None, 0, None, K, _ptr(prev_idx),
                                         _ptr(out_idx), None, _stream(stream)), "csa2_index_topk_noalloc(REUSE)")
        return out_idx
    _dev(q_idx, "q_idx", _B16)
    H_I = q_idx.shape[2]
    if q_idx.shape != (B_, T_, H_I, D_IDX):
        raise ValueError("q_idx must be [B, T, H_I, 64]")
    _dev(w_idx, "w_idx", (torch.float32,), (B_, T_, H_I))
    _dev(z, "z", _B16)
    N = z.shape[1]
    if z.shape != (B_, N, D_IDX):
        raise ValueError("z must be [B, N, 64]")
    _dev(n_visible, "n_visible", (torch.int32,), (B_ * T_,))
    if mode == REINDEX_POOL:
        if prev_idx is None:
            raise ValueError("REINDEX_POOL needs the FULL layer's selection as prev_idx")
        _dev(prev_idx, "prev_idx", (torch.int32,), (B_, T_, K))
    else:
        prev_idx = None
    if out_scores is not None:
        _dev(out_scores, "out_scores", (torch.float32,), (B_, T_, K))
    _check(L.csa2_index_topk_noalloc(mode, B_, T_, H_I, _ptr(q_idx), _ptr(w_idx), _ptr(z), N, _ptr(n_visible), K,
                                     _ptr(prev_idx), _ptr(out_idx), _ptr(out_scores), _stream(stream)),
           "csa2_index_topk_noalloc")
    return out_idx


def csa2_sparse_decode(q: torch.Tensor, kv_codes: torch.Tensor, kv_scales: torch.Tensor, idx: torch.Tensor,
                       softmax_scale: float = 1.0 / math.sqrt(D_KV), d_v: int = D_LATENT,
                       o_g: Optional[torch.Tensor] = None, lse_g: Optional[torch.Tensor] = None,
                       ws: Optional[torch.Tensor] = None, stream=None):
    """Global branch: q [B, T, H, 576] bf16 over kv_codes [B, N, 288], kv_scales [B, N, 36],
    idx [B, T, K] int32 -> (O_g [B, T, H, d_v] fp32, LSE_g [B, T, H] fp32)."""
    L = _lib()
    _dev(q, "q", _B16)
    B, T, H, _ = q.shape
    _dev_kv(kv_codes, "kv_codes", None, CODE_BYTES)
    N = kv_codes.shape[1]
    _dev_kv(kv_codes, "kv_codes", (B, N), CODE_BYTES)
    _dev_kv(kv_scales, "kv_scales", (B, N), SCALE_BYTES)
    _dev(idx, "idx", (torch.int32,))
    K = idx.shape[2]
    _dev(idx, "idx", (torch.int32,), (B, T, K))
    if o_g is None:
        o_g = torch.empty((B, T, H, d_v), dtype=torch.float32, device=q.device)
    if lse_g is None:
        lse_g = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
    _dev(o_g, "o_g", (torch.float32,), (B, T, H, d_v))
    _dev(lse_g, "lse_g", (torch.float32,), (B, T, H))
    if ws is None:
        ws = csa2_workspace(B, T, H, 0, K, device=q.device, stream=stream)
    _check(L.csa2_sparse_decode(B, T, H, _ptr(q), _ptr(kv_codes), _ptr(kv_scales), N, _ptr(idx), K, d_v,
                                float(softmax_scale), _ptr(o_g), _ptr(lse_g), _ptr(ws), ws.numel(),
                                _stream(stream)), "csa2_sparse_decode")
    return o_g, lse_g


def csa2_swa_merge(q: torch.Tensor, swa_kv: torch.Tensor, win_start: torch.Tensor, win_len: torch.Tensor,
                   n_win: int, o_g: torch.Tensor, lse_g: torch.Tensor,
                   softmax_scale: float = 1.0 / math.sqrt(D_KV), d_v: int = D_LATENT,
                   o_out: Optional[torch.Tensor] = None, lse_out: Optional[torch.Tensor] = None,
                   ws: Optional[torch.Tensor] = None, stream=None):
    """SWA branch over swa_kv [B, S, 576] bf16 rows win_start..+win_len, merged with (O_g, LSE_g)."""
    L = _lib()
    _dev(q, "q", _B16)
    B, T, H, _ = q.shape
    _dev(swa_kv, "swa_kv", _B16)
    S = swa_kv.shape[1]
    _dev(swa_kv, "swa_kv", _B16, (B, S, D_KV))
    _dev(win_start, "win_start", (torch.int32,), (B * T,))
    _dev(win_len, "win_len", (torch.int32,), (B * T,))
    _dev(o_g, "o_g", (torch.float32,), (B, T, H, d_v))
    _dev(lse_g, "lse_g", (torch.float32,), (B, T, H))
    if o_out is None:
        o_out = torch.empty((B, T, H, d_v), dtype=torch.float32, device=q.device)
    if lse_out is None:
        lse_out = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = csa2_workspace(B, T, H, 0, 1, device=q.device, stream=stream)
    _check(L.csa2_swa_merge(B, T, H, _ptr(q), _ptr(swa_kv), S, _ptr(win_start), _ptr(win_len), n_win, d_v,
                            float(softmax_scale), _ptr(o_g), _ptr(lse_g), _ptr(o_out), _ptr(lse_out), _ptr(ws),
                            ws.numel(), _stream(stream)), "csa2_swa_merge")
    return o_out, lse_out


def csa2_decode_attention(q: torch.Tensor, kv_codes: torch.Tensor, kv_scales: torch.Tensor, idx: torch.Tensor,
                          swa_kv: torch.Tensor, win_start: torch.Tensor, win_len: torch.Tensor, n_win: int,
                          softmax_scale: float = 1.0 / math.sqrt(D_KV), d_v: int = D_LATENT,
                          o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                          ws: Optional[torch.Tensor] = None, stream=None):
    """Both branches in one softmax: q [B, T, H, 576] bf16 over the selected FP4 entries
    (kv_codes [B, N, 288], kv_scales [B, N, 36], idx [B, T, K]) and the window rows of
    swa_kv [B, S, 576] -> (O [B, T, H, d_v] fp32, LSE [B, T, H] fp32)."""
    L = _lib()
    _dev(q, "q", _B16)
    B, T, H, _ = q.shape
    _dev_kv(kv_codes, "kv_codes", None, CODE_BYTES)
    N = kv_codes.shape[1]
    _dev_kv(kv_codes, "kv_codes", (B, N), CODE_BYTES)
    _dev_kv(kv_scales, "kv_scales", (B, N), SCALE_BYTES)
    _dev(idx, "idx", (torch.int32,))
    K = idx.shape[2]
    _dev(idx, "idx", (torch.int32,), (B, T, K))
    _dev(swa_kv, "swa_kv", _B16)
    S = swa_kv.shape[1]
    _dev(swa_kv, "swa_kv", _B16, (B, S, D_KV))
    _dev(win_start, "win_start", (torch.int32,), (B * T,))
    _dev(win_len, "win_len", (torch.int32,), (B * T,))
    if o is None:
        o = torch.empty((B, T, H, d_v), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
    _dev(o, "o", (torch.float32,), (B, T, H, d_v))
    _dev(lse, "lse", (torch.float32,), (B, T, H))
    if ws is None:
        ws = csa2_workspace(B, T, H, 0, K, device=q.device, stream=stream)
    _check(L.csa2_decode_attention(B, T, H, _ptr(q), _ptr(kv_codes), _ptr(kv_scales), N, _ptr(idx), K,
                                   _ptr(swa_kv), S, _ptr(win_start), _ptr(win_len), n_win, d_v,
                                   float(softmax_scale), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
                                   _stream(stream)), "csa2_decode_attention")
    return o, lse


def csa2_decode_layer(mode: int, q: torch.Tensor, kv_codes: torch.Tensor, kv_scales: torch.Tensor,
                      swa_kv: torch.Tensor, win_start: torch.Tensor, win_len: torch.Tensor, n_win: int, K: int,
                      q_idx=None, w_idx=None, z=None, n_visible=None, prev_idx=None, out_idx=None,
                      softmax_scale: float = 1.0 / math.sqrt(D_KV), d_v: int = D_LATENT,
                      o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                      ws: Optional[torch.Tensor] = None, stream=None):
    """One CSA2 decode layer in one call: the top-K selection of `mode` (as csa2_index_topk)
    and the attention over it and the window (as csa2_decode_attention). Returns
    (O [B, T, H, d_v] fp32, LSE [B, T, H] fp32, idx [B, T, K] int32)."""
    L = _lib()
    _dev(q, "q", _B16)
    B, T, H, _ = q.shape
    _dev_kv(kv_codes, "kv_codes", None, CODE_BYTES)
    N = kv_codes.shape[1]
    _dev_kv(kv_codes, "kv_codes", (B, N), CODE_BYTES)
    _dev_kv(kv_scales, "kv_scales", (B, N), SCALE_BYTES)
    _dev(swa_kv, "swa_kv", _B16)
    S = swa_kv.shape[1]
    _dev(swa_kv, "swa_kv", _B16, (B, S, D_KV))
    _dev(win_start, "win_start", (torch.int32,), (B * T,))
    _dev(win_len, "win_len", (torch.int32,), (B * T,))
    H_I = 0
    if mode in (REUSE, REINDEX_POOL):
        if prev_idx is None:
            raise ValueError("REUSE and REINDEX_POOL need prev_idx")
        _dev(prev_idx, "prev_idx", (torch.int32,), (B, T, K))
    if mode != REUSE:
        _dev(q_idx, "q_idx", _B16)
        H_I = q_idx.shape[2]
        _dev(q_idx, "q_idx", _B16, (B, T, H_I, D_IDX))
        _dev(w_idx, "w_idx", (torch.float32,), (B, T, H_I))
        _dev(z, "z", _B16, (B, N, D_IDX))
        _dev(n_visible, "n_visible", (torch.int32,), (B * T,))
    if out_idx is None:
        out_idx = torch.empty((B, T, K), dtype=torch.int32, device=q.device)
    _dev(out_idx, "out_idx", (torch.int32,), (B, T, K))
    if o is None:
        o = torch.empty((B, T, H, d_v), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
    _dev(o, "o", (torch.float32,), (B, T, H, d_v))
    _dev(lse, "lse", (torch.float32,), (B, T, H))
    if ws is None:
        ws = csa2_workspace(B, T, H, N if mode != REUSE else 0, K, device=q.device, stream=stream)
    _check(L.csa2_decode_layer(mode, B, T, H, H_I, _ptr(q), _ptr(q_idx), _ptr(w_idx), _ptr(z), _ptr(kv_codes),
                               _ptr(kv_scales), N, _ptr(n_visible), K, _ptr(prev_idx), _ptr(out_idx), _ptr(swa_kv),
                               S, _ptr(win_start), _ptr(win_len), n_win, d_v, float(softmax_scale), _ptr(o),
                               _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)), "csa2_decode_layer")
    return o, lse, out_idx


def csa2_cache_append(n_tokens: torch.Tensor, swa_row: Optional[torch.Tensor] = None,
                      swa_kv: Optional[torch.Tensor] = None, n_win: Optional[int] = None,
                      entry_kv: Optional[torch.Tensor] = None, entry_z: Optional[torch.Tensor] = None,
                      kv_codes: Optional[torch.Tensor] = None, kv_scales: Optional[torch.Tensor] = None,
                      z: Optional[torch.Tensor] = None, n_visible: Optional[torch.Tensor] = None,
                      win_start: Optional[torch.Tensor] = None, win_len: Optional[torch.Tensor] = None,
                      ratio: int = 4, advance: bool = True, ws: Optional[torch.Tensor] = None, stream=None):
    """Append one token per sequence, in place: n_tokens [B] int32 (the new token's
    position; < 0 = idle), swa_row [B, 576] bf16 into the mirrored window ring swa_kv
    [B, S >= 2 n_win, 576] (n_win defaults to S // 2), and every ratio-th token the
    compressed entry entry_kv [B, 576] (fp32/bf16, FP4-encoded into kv_codes [B, N, 288]
    / kv_scales [B, N, 36], rows ENTRY_BYTES apart as csa2_kv_cache makes them) and its
    key entry_z [B, 64] (into z [B, N, 64]); writes
    n_visible, win_start, win_len [B] int32 when given; advance increments n_tokens."""
    L = _lib()
    _dev(n_tokens, "n_tokens", (torch.int32,))
    B = n_tokens.numel()
    _dev(n_tokens, "n_tokens", (torch.int32,), (B,))
    S = 0
    if swa_kv is not None:
        _dev(swa_kv, "swa_kv", _B16)
        S = swa_kv.shape[1]
        _dev(swa_kv, "swa_kv", _B16, (B, S, D_KV))
        if n_win is None:
            n_win = S // 2
    if swa_row is not None:
        _dev(swa_row, "swa_row", _B16, (B, D_KV))
    N = 0
    if kv_codes is not None:
        _dev_kv(kv_codes, "kv_codes", None, CODE_BYTES)
        N = kv_codes.shape[1]
        _dev_kv(kv_codes, "kv_codes", (B, N), CODE_BYTES)
    if kv_scales is not None:
        _dev_kv(kv_scales, "kv_scales", (B, N), SCALE_BYTES)
    if z is not None:
        _dev(z, "z", _B16)
        if kv_codes is None:
            N = z.shape[1]
        _dev(z, "z", _B16, (B, N, D_IDX))
    dt = F32
    if entry_kv is not None:
        _dev(entry_kv, "entry_kv", (torch.float32,) + _B16, (B, D_KV))
        dt = F32 if entry_kv.dtype == torch.float32 else BF16
    if entry_z is not None:
        _dev(entry_z, "entry_z", _B16, (B, D_IDX))
    for t, name in ((n_visible, "n_visible"), (win_start, "win_start"), (win_len, "win_len")):
        if t is not None:
            _dev(t, name, (torch.int32,), (B,))
    if ws is None:
        ws = csa2_workspace(B, 1, 1, 0, 1, device=n_tokens.device, stream=stream)
    _check(L.csa2_cache_append(B, _ptr(n_tokens), 1 if advance else 0, int(ratio), _ptr(swa_row), _ptr(swa_kv), S,
                               int(n_win or 0), _ptr(entry_kv), dt, _ptr(entry_z), _ptr(kv_codes), _ptr(kv_scales),
                               _ptr(z), N, _ptr(n_visible), _ptr(win_start), _ptr(win_len), _ptr(ws), ws.numel(),
                               _stream(stream)), "csa2_cache_append")


def csa2_check_bounded_wait(limit_ns: int, ws: torch.Tensor, stream=None) -> None:
    """Run the kernels' wait-timeout path on purpose (a wait on an mbarrier nothing
    arrives on, bounded by limit_ns); read the result with csa2_read_device_status."""
    _check(_lib().csa2_check_bounded_wait(int(limit_ns), _ptr(ws), ws.numel(), _stream(stream)),
           "csa2_check_bounded_wait")


def decode_layer(mode: int, q: torch.Tensor, kv_codes: torch.Tensor, kv_scales: torch.Tensor,
                 swa_kv: torch.Tensor, win_start: torch.Tensor, win_len: torch.Tensor, n_win: int, K: int,
                 q_idx=None, w_idx=None, z=None, n_visible=None, prev_idx=None, ws=None, out_idx=None,
                 softmax_scale: float = 1.0 / math.sqrt(D_KV), fused: bool = True, stream=None):
    """One CSA2 layer: one csa2_decode_layer call (fused), or csa2_index_topk (by mode)
    followed by csa2_sparse_decode and csa2_swa_merge. Returns (O, LSE, idx)."""
    if fused:
        return csa2_decode_layer(mode, q, kv_codes, kv_scales, swa_kv, win_start, win_len, n_win, K,
                                 q_idx=q_idx, w_idx=w_idx, z=z, n_visible=n_visible, prev_idx=prev_idx,
                                 out_idx=out_idx, softmax_scale=softmax_scale, ws=ws, stream=stream)
    idx = csa2_index_topk(mode, q_idx, w_idx, z, n_visible, K, prev_idx=prev_idx, out_idx=out_idx, ws=ws,
                          stream=stream)
    o_g, lse_g = csa2_sparse_decode(q, kv_codes, kv_scales, idx, softmax_scale, ws=ws, stream=stream)
    o, lse = csa2_swa_merge(q, swa_kv, win_start, win_len, n_win, o_g, lse_g, softmax_scale, o_out=o_g,
                            lse_out=lse_g, ws=ws, stream=stream)
    return o, lse, idx
