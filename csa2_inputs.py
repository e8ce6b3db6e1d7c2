"""Seeded synthetic inputs for the CSA2 decode path and the CED KV projection.

This module is the only code shared by the CUDA path's tests/bench and the CPU
oracle. It draws random numbers and rounds them to the storage types the
workloads are defined in (bf16 by round-to-nearest-even). It contains none of
the method's arithmetic: no quantiser, no indexer, no top-K, no attention.

Workload shapes follow the synthetic configurations of this project (decode at
4K/128K/1M context, the CED projection, and a prefill chunk); the pages of
"DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" give the
dimensions used (latent 512 + rope 64, 4:1 block compression, top-K 2048,
20 decoder layers) but no data, so every input here is synthetic.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import numpy as np

FULL, REINDEX, REUSE, REINDEX_POOL = 0, 1, 2, 3
MODE_NAMES = {FULL: "FULL", REINDEX: "REINDEX", REUSE: "REUSE", REINDEX_POOL: "REINDEX_POOL"}

D_LATENT = 512
D_ROPE = 64
D_KV = D_LATENT + D_ROPE  # 576
D_IDX = 64
COMPRESS = 4  # raw tokens per compressed entry


# ----------------------------------------------------------------------------
# bf16 storage helpers (input preparation only)
# ----------------------------------------------------------------------------
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (nearest, ties to even); return the uint16 bit patterns.

    For finite inputs u + 0x7FFF + lsb stays below 2^32, so uint32 arithmetic is exact."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.reshape(-1).view(np.uint32)
    out = np.empty(u.shape, dtype=np.uint16)
    step = 1 << 22
    for i in range(0, u.size, step):
        c = u[i:i + step]
        r = c + np.uint32(0x7FFF)
        r += (c >> np.uint32(16)) & np.uint32(1)
        out[i:i + step] = r >> np.uint32(16)
    return out.reshape(x.shape)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to the fp32 values they denote."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# Configurations
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class DecodeConfig:
    """One decode (T=1) or prefill-chunk (T>1) workload over a compressed KV cache.

    N is the number of compressed entries per sequence (context / 4). The query
    tokens sit at the end of the context: token positions ctx-T .. ctx-1.
    """
    name: str
    B: int
    T: int
    N: int
    H: int
    H_I: int
    K: int
    W: int
    modes: Tuple[int, ...]
    seed: int
    planted_bias: float = 0.0   # rank-1 recency bias added to indexer keys
    causal: bool = False        # per-query visibility of compressed entries
    d_v: int = D_LATENT

    @property
    def ctx(self) -> int:
        return COMPRESS * self.N

    @property
    def positions(self) -> np.ndarray:
        return np.arange(self.ctx - self.T, self.ctx, dtype=np.int64)

    @property
    def S(self) -> int:
        """Rows of the raw sliding-window store per sequence."""
        return self.T + self.W - 1 if self.T > 1 else self.W

    @property
    def softmax_scale(self) -> float:
        return 1.0 / float(np.sqrt(D_KV))


@dataclass(frozen=True)
class CedConfig:
    """CED prefill KV projection: H [rows x d_model] times per-layer W^KV, W^Z."""
    name: str
    rows: int
    d_model: int
    n_layers: int
    seed: int


TINY = DecodeConfig("tiny_decode_b1_n1024", B=1, T=1, N=1024, H=16, H_I=4, K=128, W=128,
                    modes=(FULL,), seed=0)
DECODE_128K = DecodeConfig("decode_b32_ctx128k_full_reindex_reuse", B=32, T=1, N=32768, H=64,
                           H_I=8, K=2048, W=128, modes=(FULL, REINDEX, REUSE), seed=1,
                           planted_bias=3.0)
DECODE_1M = DecodeConfig("decode_b4_ctx1m_full", B=4, T=1, N=262144, H=64, H_I=8, K=2048,
                         W=128, modes=(FULL,), seed=2)
CED_PROJ = CedConfig("ced_projection_32768x4096_20layers", rows=32768, d_model=4096,
                     n_layers=20, seed=3)
PREFILL_CHUNK = DecodeConfig("prefill_chunk_t4096_ctx128k", B=1, T=4096, N=32768, H=64, H_I=8,
                             K=2048, W=128, modes=(FULL,), seed=4, causal=True)

CONFIGS = {c.name: c for c in (TINY, DECODE_128K, DECODE_1M, CED_PROJ, PREFILL_CHUNK)}


def scaled(cfg: DecodeConfig, **kw) -> DecodeConfig:
    """Same workload recipe at other sizes (for parity tests that must stay small)."""
    d = dict(cfg.__dict__)
    d.update(kw)
    if "name" not in kw:
        d["name"] = cfg.name + "_scaled"
    return DecodeConfig(**d)


# ----------------------------------------------------------------------------
# Generated tensors
# ----------------------------------------------------------------------------
@dataclass
class LayerInputs:
    mode: int
    X: Optional[np.ndarray]        # fp32 [B, N, 576] latent KV before FP4 encode (FULL only)
    z: Optional[np.ndarray]        # bf16 bits [B, N, 64] indexer keys (FULL, REINDEX)
    q_idx: Optional[np.ndarray]    # bf16 bits [B, T, H_I, 64]
    w_idx: Optional[np.ndarray]    # fp32 [B, T, H_I]
    q: np.ndarray                  # bf16 bits [B, T, H, 576]
    swa: np.ndarray                # bf16 bits [B, S, 576]


@dataclass
class DecodeInputs:
    cfg: DecodeConfig
    layers: List[LayerInputs]
    n_visible: np.ndarray          # int32 [B*T]
    win_start: np.ndarray          # int32 [B*T]
    win_len: np.ndarray            # int32 [B*T]
    extra: Dict[str, np.ndarray] = field(default_factory=dict)


def visibility(cfg: DecodeConfig) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Per-query number of visible entries and the sliding-window rows.

    An entry j summarises raw tokens [4j, 4j+3]; a query at token position p
    sees it iff 4j+3 <= p. Decode queries (T=1) see all N entries. The window is
    the last min(W, p+1) raw tokens up to and including p.
    """
    pos = cfg.positions
    if cfg.causal:
        nvis = (pos + 1) // COMPRESS
    else:
        nvis = np.full(cfg.T, cfg.N, dtype=np.int64)
    wlen = np.minimum(cfg.W, pos + 1)
    if cfg.T > 1:
        # store row r holds token position pos[0] - (W-1) + r
        wstart = np.arange(cfg.T, dtype=np.int64) + (cfg.W - wlen)
    else:
        wstart = np.full(cfg.T, cfg.W, dtype=np.int64) - wlen
    rep = lambda a: np.tile(a.astype(np.int32), cfg.B)
    return rep(nvis), rep(wstart), rep(wlen)


def _stream(seed: int, *key: int) -> np.random.Generator:
    """Independent PCG64 stream for one tensor, keyed by (seed, layer, tensor tag)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


_TAG = {"u": 0, "X": 1, "z": 2, "q_idx": 3, "w_idx": 4, "q": 5, "swa": 6}


def _per_sequence_normal(seed: int, layer: int, tag: int, B: int, shape) -> np.ndarray:
    """fp32 N(0,1) array [B, *shape]; sequence b drawn from stream (seed, layer, tag, b).

    Sequences are drawn on a thread pool (NumPy releases the GIL while filling)."""
    from concurrent.futures import ThreadPoolExecutor
    import os
    out = np.empty((B,) + tuple(shape), dtype=np.float32)

    def fill(b):
        _stream(seed, layer, tag, b).standard_normal(tuple(shape), dtype=np.float32, out=out[b])

    n = min(B, max(1, len(os.sched_getaffinity(0))))
    if n == 1:
        for b in range(B):
            fill(b)
    else:
        with ThreadPoolExecutor(n) as ex:
            list(ex.map(fill, range(B)))
    return out


def make_decode_inputs(cfg: DecodeConfig, with_x: bool = True) -> DecodeInputs:
    """Draw every input of a decode group; each tensor has its own PCG64 stream.

    Per layer: X (FULL only), z (FULL, REINDEX), q_idx, w_idx (FULL, REINDEX), q, swa;
    X and z have one stream per sequence.
    Every draw is standard normal in fp32; w_idx takes absolute values; every
    bf16 tensor is rounded to nearest-even. With planted_bias > 0 a unit vector
    u is drawn and keys get z[b, n] += bias * n/(N-1) * u, which makes the
    indexer prefer recent entries for heads aligned with u. with_x=False skips
    the fp32 latent KV (the other tensors are unchanged, their streams being
    independent).
    """
    B, T, N, H, H_I = cfg.B, cfg.T, cfg.N, cfg.H, cfg.H_I
    u = None
    if cfg.planted_bias:
        u = _stream(cfg.seed, 0, _TAG["u"]).standard_normal(D_IDX, dtype=np.float32)
        u = (u / np.linalg.norm(u)).astype(np.float32)
    layers: List[LayerInputs] = []
    for li, mode in enumerate(cfg.modes):
        X = z = q_idx = w_idx = None
        if mode == FULL and with_x:
            X = _per_sequence_normal(cfg.seed, li, _TAG["X"], B, (N, D_KV))
        if mode in (FULL, REINDEX):
            zf = _per_sequence_normal(cfg.seed, li, _TAG["z"], B, (N, D_IDX))
            if u is not None:
                ramp = (np.arange(N, dtype=np.float32) / np.float32(max(N - 1, 1)))
                zf += (np.float32(cfg.planted_bias) * ramp)[None, :, None] * u[None, None, :]
            z = bf16_bits(zf)
            del zf
            q_idx = bf16_bits(_stream(cfg.seed, li, _TAG["q_idx"]).standard_normal((B, T, H_I, D_IDX),
                                                                                    dtype=np.float32))
            w_idx = np.abs(_stream(cfg.seed, li, _TAG["w_idx"]).standard_normal((B, T, H_I), dtype=np.float32))
        q = bf16_bits(_stream(cfg.seed, li, _TAG["q"]).standard_normal((B, T, H, D_KV), dtype=np.float32))
        swa = bf16_bits(_stream(cfg.seed, li, _TAG["swa"]).standard_normal((B, cfg.S, D_KV), dtype=np.float32))
        layers.append(LayerInputs(mode, X, z, q_idx, w_idx, q, swa))
    nvis, wstart, wlen = visibility(cfg)
    return DecodeInputs(cfg, layers, nvis, wstart, wlen)


def latent_rows(cfg: DecodeConfig, layer: int, b: int, rows: np.ndarray) -> np.ndarray:
    """Rows of the FULL layer's fp32 latent KV for one sequence (regenerated from its stream)."""
    X = _stream(cfg.seed, layer, _TAG["X"], b).standard_normal((cfg.N, D_KV), dtype=np.float32)
    return X[rows]


@dataclass
class CedInputs:
    cfg: CedConfig
    H: np.ndarray      # bf16 bits [rows, d_model]
    W_kv: np.ndarray   # bf16 bits [n_layers, 576, d_model] (row c = weights of output channel c)
    W_z: np.ndarray    # bf16 bits [n_layers, 64, d_model]


def make_ced_inputs(cfg: CedConfig) -> CedInputs:
    """H ~ N(0,1)/64 and W ~ N(0, 1/d_model), all rounded to bf16 (one stream per tensor)."""
    Hm = bf16_bits(_stream(cfg.seed, 0, 0).standard_normal((cfg.rows, cfg.d_model), dtype=np.float32)
                   / np.float32(64))
    ws = np.float32(1.0 / np.sqrt(cfg.d_model))
    Wkv = bf16_bits(_stream(cfg.seed, 0, 1).standard_normal((cfg.n_layers, D_KV, cfg.d_model),
                                                            dtype=np.float32) * ws)
    Wz = bf16_bits(_stream(cfg.seed, 0, 2).standard_normal((cfg.n_layers, D_IDX, cfg.d_model),
                                                           dtype=np.float32) * ws)
    return CedInputs(cfg, Hm, Wkv, Wz)


def encode_rows_input(rows: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """fp32 [rows, 576] N(0, scale^2) rows for quantise-only encode tests."""
    return _stream(seed, 0, 0).standard_normal((rows, D_KV), dtype=np.float32) * np.float32(scale)
