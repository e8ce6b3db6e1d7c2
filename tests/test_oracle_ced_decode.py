"""Pins of the oracle's CED projection and of the layer-mode semantics (no GPU).

Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", picx.dev summary,
Methodology / 1. CED, Eq. (1), and / 2. CSA2 (FULL, REINDEX, REUSE).
"""
from fractions import Fraction

import numpy as np

import csa2_inputs as ci
from oracle import attention, ced, decode, fp4


def test_projection_of_basis_rows_picks_weight_columns():
    """H = e_k gives C = W^KV[k, :] (row k of W^KV, i.e. column k of the stored W^T):
    catches a transposed or mis-indexed operand."""
    rng = np.random.default_rng(9)
    d = 32
    Wkv = rng.standard_normal((576, d))
    Wz = rng.standard_normal((64, d))
    Hm = np.eye(d)[[3, 17]]
    C, Z = ced.project(Hm, Wkv, Wz)
    assert np.array_equal(C, Wkv[:, [3, 17]].T) and np.array_equal(Z, Wz[:, [3, 17]].T)


def test_projection_brute_force_loops():
    rng = np.random.default_rng(10)
    Hm = rng.standard_normal((3, 5)); Wkv = rng.standard_normal((576, 5)); Wz = rng.standard_normal((64, 5))
    C, Z = ced.project(Hm, Wkv, Wz)
    for r in range(3):
        for c in (0, 100, 575):
            assert np.isclose(C[r, c], sum(Hm[r, k] * Wkv[c, k] for k in range(5)), atol=1e-14)
        for c in (0, 63):
            assert np.isclose(Z[r, c], sum(Hm[r, k] * Wz[c, k] for k in range(5)), atol=1e-14)


def _bf16_by_fractions(v: float) -> float:
    f = Fraction(v)
    if f == 0:
        return 0.0
    e = abs(f).numerator.bit_length() - abs(f).denominator.bit_length()
    while Fraction(2) ** e > abs(f):
        e -= 1
    while Fraction(2) ** (e + 1) <= abs(f):
        e += 1
    ulp = Fraction(2) ** (e - 7)
    q, r = divmod(abs(f), ulp)
    if r > ulp / 2 or (r == ulp / 2 and q % 2 == 1):
        q += 1
    return float((q * ulp) * (1 if f > 0 else -1))


def test_bf16_rounding_against_exact_arithmetic():
    rng = np.random.default_rng(11)
    vals = list(rng.standard_normal(300) * 10 ** rng.uniform(-5, 5, 300))
    vals += [1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 255.5, 256.5, 1 - 2 ** -10]
    for v in vals:
        assert ced.to_bf16_rne(np.array([v]))[0] == _bf16_by_fractions(float(v)), v


def test_ambiguity_bound_covers_fp32_summation():
    rng = np.random.default_rng(12)
    Hm = rng.standard_normal((4, 4096)).astype(np.float32) / 64
    W = (rng.standard_normal((8, 4096)) / 64).astype(np.float32)
    exact = Hm.astype(np.float64) @ W.astype(np.float64).T
    naive = np.zeros((4, 8), dtype=np.float32)
    for k in range(4096):
        naive += Hm[:, k:k + 1] * W[:, k][None, :]
    assert np.all(np.abs(naive - exact) <= ced.ambiguity_bound(Hm, W))


def _small_group():
    cfg = ci.scaled(ci.DECODE_128K, B=2, N=96, H=4, H_I=2, K=16, W=8)
    return cfg, ci.make_decode_inputs(cfg)


def _run(cfg, inp):
    f64 = lambda b: ci.bf16_bits_to_f32(b).astype(np.float64)
    return [decode.run_group_sequence(inp.layers, b, inp.n_visible, inp.win_start, inp.win_len,
                                      cfg.K, cfg.d_v, cfg.softmax_scale, f64) for b in range(cfg.B)]


def test_modes_reuse_and_reindex_semantics():
    cfg, inp = _small_group()
    before = [L.X.copy() if L.X is not None else None for L in inp.layers]
    res = _run(cfg, inp)
    for b in range(cfg.B):
        full, reindex, reuse = res[b]
        # REINDEX and REUSE read the FULL layer's KV bytes unchanged
        assert reindex["codes"] is full["codes"] and reuse["codes"] is full["codes"]
        # REINDEX computes fresh indices (its own indexer differs), REUSE repeats them exactly
        assert not np.array_equal(reindex["idx"], full["idx"])
        assert np.array_equal(reuse["idx"], reindex["idx"])
    for L, x0 in zip(inp.layers, before):
        if x0 is not None:
            assert np.array_equal(L.X, x0)


def test_full_with_k_ge_n_is_dense_over_entries_and_window():
    cfg = ci.scaled(ci.TINY, N=24, H=2, H_I=2, K=32, W=8)
    inp = ci.make_decode_inputs(cfg)
    f64 = lambda b: ci.bf16_bits_to_f32(b).astype(np.float64)
    r = decode.run_group_sequence(inp.layers, 0, inp.n_visible, inp.win_start, inp.win_len,
                                  cfg.K, cfg.d_v, cfg.softmax_scale, f64)[0]
    L = inp.layers[0]
    rows = fp4.decode(*fp4.encode(L.X[0]))
    union = np.vstack([rows, f64(L.swa[0])])
    O, lse = attention.attend(f64(L.q[0])[0], union, cfg.d_v, cfg.softmax_scale)
    assert np.allclose(r["O"][0], O, atol=1e-12) and np.allclose(r["LSE"][0], lse, atol=1e-12)
