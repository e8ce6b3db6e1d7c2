"""Shared test helpers: device upload of generated inputs and parity comparisons."""
from __future__ import annotations

import numpy as np

import csa2_inputs as ci

# Tolerances fixed by the benchmark spec for the attention outputs.
ATOL_MAX_ABS = 2e-3
RTOL_REL_L2 = 1e-3
TIE_REL = 1e-6


def f64(bits: np.ndarray) -> np.ndarray:
    return ci.bf16_bits_to_f32(bits).astype(np.float64)


def to_dev_bf16(bits: np.ndarray, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def to_dev(a: np.ndarray, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def check_index_set(got: np.ndarray, want: np.ndarray, scores: np.ndarray, n_visible: int, K: int):
    """GPU and oracle top-K sets agree, except entries whose oracle score is within
    1e-6 relative of the K-th score. Also: sorted ascending, -1 padded, no repeats."""
    from oracle import indexer
    g = got[got >= 0]
    assert np.all(np.diff(g) > 0), "indices must be strictly ascending"
    assert g.size == min(K, n_visible), (g.size, min(K, n_visible))
    assert np.all(got[g.size:] == -1)
    assert np.all(g < n_visible)
    kth = indexer.kth_score(scores, n_visible, K)
    diff = np.setxor1d(g, want[want >= 0])
    if diff.size:
        tol = TIE_REL * abs(kth)
        bad = diff[np.abs(scores[diff] - kth) > tol]
        assert bad.size == 0, f"{bad.size} index-set differences outside the tie band (kth={kth})"
    return int(diff.size)


def check_attention(got: np.ndarray, want: np.ndarray, what: str = ""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want).max() if got.size else 0.0
    den = np.linalg.norm(want)
    rel = np.linalg.norm(got - want) / den if den > 0 else np.linalg.norm(got)
    assert err <= ATOL_MAX_ABS and rel <= RTOL_REL_L2, f"{what}: max-abs {err:.3e}, rel-L2 {rel:.3e}"
    return err, rel


def check_lse(got: np.ndarray, want: np.ndarray, what: str = ""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    inf_g, inf_w = np.isneginf(got), np.isneginf(want)
    assert np.array_equal(inf_g, inf_w), f"{what}: -inf pattern differs"
    m = ~inf_w
    if m.any():
        err = np.abs(got[m] - want[m]).max()
        assert err <= ATOL_MAX_ABS, f"{what}: LSE max-abs {err:.3e}"
