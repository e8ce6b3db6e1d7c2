"""FP4 quantiser parity: CUDA codes and scales are bit-exact with the oracle.

Format: E2M1 with one E4M3 scale per 16 channels ("DeepSeek-V4.1-Flash: Pushing the
Limits of KV Cache Compression", picx.dev summary, Methodology / 5. FP4 Main KV Cache).
"""
import numpy as np
import pytest
import torch

import csa2_inputs as ci
from oracle import fp4
from tests._util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    import sparse_attention_kv_decode_b300 as m
    m.lib()
    return m


def _gpu_encode(csa2, x32: np.ndarray):
    c, s = csa2.csa2_encode_kv(to_dev(x32, "cuda"))
    torch.cuda.synchronize()
    return c.cpu().numpy(), s.cpu().numpy()


def _assert_same(csa2, x32):
    gc, gs = _gpu_encode(csa2, x32)
    oc, os_ = fp4.encode(x32.reshape(-1, 576))
    assert np.array_equal(gs.reshape(os_.shape), os_), "scale codes differ"
    bad = np.nonzero((gc.reshape(oc.shape) != oc).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows with differing codes, first {bad[:5]}"


def test_random_rows_fp32(csa2):
    x = ci.encode_rows_input(4099, seed=11)          # ragged count of rows
    _assert_same(csa2, x)


def test_small_magnitudes_subnormal_scales(csa2):
    # config-4-like magnitudes put amax/6 in the E4M3 subnormal range
    x = ci.encode_rows_input(2048, seed=12, scale=1.0 / 64)
    _assert_same(csa2, x)
    x = ci.encode_rows_input(512, seed=13, scale=1e-3)
    _assert_same(csa2, x)


def test_bf16_input_matches_widened_fp32(csa2):
    x = ci.encode_rows_input(1000, seed=14)
    bits = ci.bf16_bits(x)
    xb = ci.bf16_bits_to_f32(bits)
    t = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    c, s = csa2.csa2_encode_kv(t)
    oc, os_ = fp4.encode(xb)
    assert np.array_equal(c.cpu().numpy(), oc) and np.array_equal(s.cpu().numpy(), os_)


def _boundary_rows():
    """Blocks whose elements sit on every E2M1 midpoint (and one ulp either side), for
    scales across the E4M3 range, plus blocks whose amax/6 sits on E4M3 midpoints."""
    rows = []
    mids = [(a + b) / 2 for a, b in zip(fp4.E2M1_MAG[:-1], fp4.E2M1_MAG[1:])] + [6.0, 6.5, 7.0]
    for scode in [0x01, 0x03, 0x07, 0x08, 0x20, 0x38, 0x50, 0x7E]:
        s = float(fp4.e4m3_value(scode))
        for d in (-1, 0, 1):
            vals = []
            for m in mids:
                v = np.float32(m * s)
                if d:
                    v = np.nextafter(v, np.float32(d * np.inf))
                vals.append(v)
            blk = np.array(vals[:10] + [-v for v in vals[:5]] + [np.float32(6 * s)], dtype=np.float32)
            rows.append(blk)
    for a, b in zip(fp4.E4M3_POS[:-1], fp4.E4M3_POS[1:]):
        m = np.float32((a + b) / 2 * 6)
        for v in (np.nextafter(m, np.float32(0)), m, np.nextafter(m, np.float32(np.inf))):
            blk = np.linspace(-1, 1, 16, dtype=np.float32) * v
            rows.append(blk.astype(np.float32))
    blocks = np.stack(rows)
    pad = (-len(blocks)) % 36
    blocks = np.concatenate([blocks, np.zeros((pad, 16), np.float32)])
    return blocks.reshape(-1, 576)


def test_rounding_boundaries_bit_exact(csa2):
    _assert_same(csa2, _boundary_rows())


def test_saturation_and_zero_blocks(csa2):
    x = np.zeros((2, 576), np.float32)
    x[0, :16] = np.linspace(-1e6, 1e6, 16)
    x[0, 16:32] = 6 * 2.0 ** -11
    x[1, :] = -0.0
    _assert_same(csa2, x)


def test_full_size_launch_sampled(csa2):
    """The decode cache's launch shape (32 sequences x 32768 entries would be 1M rows);
    here 262144 rows through the same grid-stride kernel, checked on a sample."""
    x = ci.encode_rows_input(262144, seed=15)
    gc, gs = _gpu_encode(csa2, x)
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(x.shape[0], 4096, replace=False))
    rows = np.concatenate([rows, [0, x.shape[0] - 1]])
    oc, os_ = fp4.encode(x[rows])
    assert np.array_equal(gc[rows], oc) and np.array_equal(gs[rows], os_)


def test_deterministic(csa2):
    x = ci.encode_rows_input(777, seed=16)
    a = _gpu_encode(csa2, x)
    b = _gpu_encode(csa2, x)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
