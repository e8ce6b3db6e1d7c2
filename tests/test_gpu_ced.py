"""CED projection (Eq. (1)) with the fused FP4 cache write: parity with the FP64 oracle.

Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", picx.dev summary,
Methodology / 1. CED, Eq. (1), and / 5. FP4 Main KV Cache.

The device accumulates the product in fp32 on the tensor cores; the oracle computes it
exactly. A 16-channel block is "boundary-ambiguous" when the exact value's scale or any
code could round differently anywhere inside the fp32 accumulation error bound
(gamma_d * sum|h||w|); every other block must match the oracle bit for bit, and the
ambiguous ones must still satisfy the quantiser's error bound. Z is within 1 bf16 ulp.
"""
import numpy as np
import pytest
import torch

import csa2_inputs as ci
import sparse_attention_kv_decode_b300 as csa2
from oracle import ced, fp4
from tests._util import f64, to_dev_bf16

pytestmark = pytest.mark.gpu


def _run(inp):
    h = to_dev_bf16(inp.H, "cuda")
    wkv = to_dev_bf16(inp.W_kv, "cuda")
    wz = to_dev_bf16(inp.W_z, "cuda")
    ws = csa2.csa2_workspace(0, 0, 0, 0, 0)
    codes, scales, z = csa2.csa2_encode_kv(h, wkv, wz, ws=ws)
    torch.cuda.synchronize()
    st, flags = csa2.csa2_read_device_status(ws)
    assert st == 0, (st, flags)
    return codes.cpu().numpy(), scales.cpu().numpy(), z.view(torch.int16).cpu().numpy().view(np.uint16)


def _check_layer(Hrows, Wkv_l, Wz_l, gc, gs, gz):
    """Compare one layer's rows. Returns the number of ambiguous blocks."""
    C, Z = ced.project(Hrows, Wkv_l, Wz_l)
    E = ced.ambiguity_bound(Hrows, Wkv_l)
    oc, osc, oz, C32 = ced.project_and_encode(Hrows, Wkv_l, Wz_l)
    R = C.shape[0]
    Cb, Eb = C.reshape(R, 36, 16), E.reshape(R, 36, 16)
    amax = np.abs(Cb).max(axis=2)
    emax = Eb.max(axis=2)
    s_lo = fp4.e4m3_encode_nonneg(np.maximum(amax - emax, 0) / 6)
    s_hi = fp4.e4m3_encode_nonneg((amax + emax) / 6)
    s_val = fp4.e4m3_value(osc).astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        c_lo = fp4.e2m1_encode(((Cb - Eb) / s_val[:, :, None]).astype(np.float32))
        c_hi = fp4.e2m1_encode(((Cb + Eb) / s_val[:, :, None]).astype(np.float32))
    code_amb = (c_lo != c_hi).any(axis=2) & (s_val > 0)
    amb = (s_lo != s_hi) | code_amb
    gcodes = fp4.unpack_codes(gc).reshape(R, 36, 16)
    ocodes = fp4.unpack_codes(oc).reshape(R, 36, 16)
    ok = ~amb
    assert np.array_equal(gs[ok], osc[ok]), "scale differs in an unambiguous block"
    assert np.array_equal(gcodes[ok], ocodes[ok]), "codes differ in an unambiguous block"
    if amb.any():
        d = fp4.decode(gc, gs).reshape(R, 36, 16)
        sv = fp4.e4m3_value(gs)[:, :, None]
        bound = sv + np.maximum(0, amax[:, :, None] - 6 * sv) + Eb
        assert np.all(np.abs(d - Cb)[amb] <= bound[amb] + 1e-12)
    # Z: the device rounds its fp32 product (within Ez of the exact Z) to bf16, so it is
    # within Ez + one bf16 ulp of |Z| + Ez of the exact value; away from cancellation this
    # is within 1 ulp of the correctly rounded bf16 value.
    zg = f64(gz)
    Ez = ced.ambiguity_bound(Hrows, Wz_l)
    ulp = np.ldexp(1.0, np.frexp(np.abs(Z) + Ez)[1] - 8)
    viol = np.abs(zg - Z) - (Ez + ulp)
    assert np.all(viol <= 0), f"Z: worst excess {viol.max():.3e} at |Z|={np.abs(Z).flat[viol.argmax()]:.3e}"
    far = Ez < ulp / 4
    ulp_r = np.ldexp(1.0, np.frexp(np.abs(oz))[1] - 8)
    assert np.all((np.abs(zg - oz) <= ulp_r)[far]), "Z off by more than 1 bf16 ulp away from cancellation"
    return int(amb.sum())


def _check_all(inp, gc, gs, gz, rows=None):
    cfg = inp.cfg
    Hf = f64(inp.H)
    rows = np.arange(cfg.rows) if rows is None else rows
    namb = 0
    for l in range(cfg.n_layers):
        namb += _check_layer(Hf[rows], f64(inp.W_kv[l]), f64(inp.W_z[l]), gc[l][rows], gs[l][rows], gz[l][rows])
    return namb


@pytest.mark.parametrize("rows,d_model,n_layers", [(256, 128, 3), (200, 192, 1), (130, 64, 2), (384, 512, 5)])
def test_small_shapes(rows, d_model, n_layers):
    cfg = ci.CedConfig("t", rows=rows, d_model=d_model, n_layers=n_layers, seed=7)
    inp = ci.make_ced_inputs(cfg)
    gc, gs, gz = _run(inp)
    _check_all(inp, gc, gs, gz)


def test_unit_scale_inputs_exercise_normal_scales():
    """N(0,1) inputs put scales in the normal E4M3 range (the config-4 magnitudes give
    subnormal scales, covered by the other tests)."""
    cfg = ci.CedConfig("t", rows=256, d_model=256, n_layers=2, seed=8)
    inp = ci.make_ced_inputs(cfg)
    inp.H = ci.bf16_bits(ci.bf16_bits_to_f32(inp.H) * 64)
    gc, gs, gz = _run(inp)
    _check_all(inp, gc, gs, gz)


def test_full_depth_k4096_twenty_layers():
    cfg = ci.CedConfig("t", rows=512, d_model=4096, n_layers=20, seed=9)
    inp = ci.make_ced_inputs(cfg)
    gc, gs, gz = _run(inp)
    namb = _check_all(inp, gc, gs, gz)
    print("ambiguous blocks:", namb, "of", 512 * 20 * 36)


def test_full_size_sampled():
    """32768 x 4096 times 20 layers x 640 (the bench shape); 96 sampled rows, all layers."""
    cfg = ci.CED_PROJ
    inp = ci.make_ced_inputs(cfg)
    gc, gs, gz = _run(inp)
    rng = np.random.default_rng(1)
    rows = np.sort(np.concatenate([rng.choice(cfg.rows, 94, replace=False), [0, cfg.rows - 1]]))
    namb = _check_all(inp, gc, gs, gz, rows=rows)
    print("ambiguous blocks:", namb, "of", rows.size * 20 * 36)


def test_deterministic():
    cfg = ci.CedConfig("t", rows=384, d_model=256, n_layers=3, seed=10)
    inp = ci.make_ced_inputs(cfg)
    a = _run(inp)
    b = _run(inp)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
