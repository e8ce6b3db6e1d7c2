"""Pins of the oracle's FP4 codec to the format definitions (no GPU).

Format: E2M1 elements with one E4M3 scale per 16 channels and range 2688 = 6*448
("DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", picx.dev summary,
Methodology / 5. FP4 Main KV Cache). Each test checks the oracle against something
other than itself: a hand-derived fixture, exact rational arithmetic, or a closed form.
"""
import os
from fractions import Fraction

import numpy as np

from oracle import fp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp4_row64.txt")


def _load_golden():
    xs, codes, scales, head = [], None, None, None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = line.split(":", 1)
        if key == "x":
            xs += [float(v) for v in val.split()]
        elif key == "codes":
            codes = bytes(int(v, 16) for v in val.split())
        elif key == "scales":
            scales = bytes(int(v, 16) for v in val.split())
        elif key == "decoded_block2_head":
            head = [float(v) for v in val.split()]
    return np.array(xs, dtype=np.float32)[None, :], codes, scales, head


def test_golden_row_hand_derived():
    x, codes, scales, head = _load_golden()
    c, s = fp4.encode(x)
    assert bytes(c[0]) == codes
    assert bytes(s[0]) == scales
    d = fp4.decode(c, s)
    assert list(d[0, 32:34]) == head


def test_format_constants_from_definition():
    # E4M3 (FN): max 1.75*2^8, min normal 2^-6, min subnormal 2^-9; E2M1 max 6.
    assert fp4.E4M3_MAX == 448.0
    assert fp4.e4m3_value(0x08) == 2.0 ** -6
    assert fp4.e4m3_value(0x01) == 2.0 ** -9
    assert fp4.e4m3_value(0x38) == 1.0
    assert np.isnan(fp4.e4m3_value(0x7F)) and np.isnan(fp4.e4m3_value(0xFF))
    assert fp4.E2M1_MAX * fp4.E4M3_MAX == 2688.0        # the range the page states
    assert np.all(np.diff(fp4.E4M3_POS) > 0) and fp4.E4M3_POS.size == 127
    assert list(fp4.e2m1_value(np.arange(16))) == [0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6]


def test_roundtrip_every_scale_code():
    """x = s * e2m1(c) with one element at +-6s encodes back to exactly (c, s) for every
    non-zero finite E4M3 scale s, normal and subnormal."""
    rng = np.random.default_rng(0)
    scodes = np.arange(1, 0x7F)
    R = scodes.size * 8
    s_code = np.repeat(scodes, 8)
    codes = rng.integers(0, 16, size=(R, 16))
    codes[codes == 8] = 0                               # -0 is stored as +0
    pos = rng.integers(0, 16, size=R)
    codes[np.arange(R), pos] = np.where(rng.random(R) < 0.5, 7, 15)   # +-6 sets amax = 6s
    s_val = fp4.e4m3_value(s_code)
    x = (fp4.e2m1_value(codes) * s_val[:, None]).astype(np.float32)
    assert np.all(x.astype(np.float64) == fp4.e2m1_value(codes) * s_val[:, None])   # exact in fp32
    got_codes, got_s = fp4.quantize_blocks(x)
    assert np.array_equal(got_s[:, 0], s_code)
    assert np.array_equal(got_codes, codes)


def _nearest_fraction(v: Fraction, table, even_of):
    best = None
    for i, t in enumerate(table):
        d = abs(v - t)
        if best is None or d < best[0] or (d == best[0] and even_of(i) and not even_of(best[1])):
            best = (d, i)
    if v >= table[-1]:
        return len(table) - 1
    return best[1]


def _neighbours(v: float):
    f = np.float32(v)
    return [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]


def test_e2m1_rounding_brute_force_at_every_midpoint():
    mags = [Fraction(m).limit_denominator() for m in fp4.E2M1_MAG]
    probes = []
    for a, b in zip(fp4.E2M1_MAG[:-1], fp4.E2M1_MAG[1:]):
        probes += _neighbours((a + b) / 2) + _neighbours(a) + _neighbours(b)
    probes += _neighbours(6.0) + [np.float32(7.0), np.float32(1e30)]
    probes = [p for p in probes if p >= 0]
    for p in probes:
        for sign in (1, -1):
            v = np.float32(sign * p)
            want_mag = _nearest_fraction(abs(Fraction(float(v))), mags, lambda i: i % 2 == 0)
            want = want_mag | (8 if (v < 0 and want_mag != 0) else 0)
            assert fp4.e2m1_encode(np.array([v]))[0] == want, (v, want)


def test_e4m3_rounding_brute_force_at_every_midpoint():
    table = [Fraction(float(t)) for t in fp4.E4M3_POS]
    probes = []
    for a, b in zip(fp4.E4M3_POS[:-1], fp4.E4M3_POS[1:]):
        probes += _neighbours((a + b) / 2)
    probes += _neighbours(448.0) + _neighbours(464.0) + [np.float32(1e6)]
    for p in probes:
        if p < 0:
            continue
        want = _nearest_fraction(Fraction(float(p)), table, lambda i: i % 2 == 0)
        assert fp4.e4m3_encode_nonneg(np.array([p]))[0] == want, (p, want)


def test_scale_underflow_boundary():
    # amax/6 == 2^-10 is the midpoint between 0 and 2^-9: ties to the even code 0.
    x = np.zeros((1, 16), dtype=np.float32)
    x[0, 3] = 6 * 2.0 ** -10
    c, s = fp4.encode(x)
    assert s[0, 0] == 0 and not c.any()
    x[0, 3] = np.nextafter(np.float32(6 * 2.0 ** -10), np.float32(1))
    c, s = fp4.encode(x)
    # the scale rounds up to 2^-9 = amax/3, so the element lands on E2M1 3.0 (code 5)
    assert s[0, 0] == 1 and fp4.unpack_codes(c)[0, 3] == 5


def test_negative_values_rounding_to_zero_store_plus_zero():
    x = np.full((1, 16), -1e-3, dtype=np.float32)
    x[0, 0] = 6.0
    c, _ = fp4.encode(x)
    assert np.all(fp4.unpack_codes(c)[0, 1:] == 0)


def test_saturation_reaches_stated_range():
    x = np.zeros((1, 16), dtype=np.float32)
    x[0, 0] = 1e9
    x[0, 1] = -3000.0
    d = fp4.decode(*fp4.encode(x))
    assert d[0, 0] == 2688.0 and d[0, 1] == -2688.0


def test_error_bound_property_on_random_rows():
    """|x - dequant(x)| <= s (half the widest E2M1 gap, 2, times s) plus the scale's rounding."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((256, 576)).astype(np.float32) * 3
    c, s = fp4.encode(x)
    d = fp4.decode(c, s)
    sv = fp4.e4m3_value(s).repeat(16, axis=1)
    amax = np.abs(x.reshape(256, 36, 16)).max(axis=2).repeat(16, axis=1)
    # values above 6s saturate; s >= amax/6 * (1 - 2^-4) after E4M3 rounding
    bound = sv + np.maximum(0, amax - 6 * sv)
    assert np.all(np.abs(x - d) <= bound + 1e-12)
    # norm bound from the page: |KV| <= sqrt(512) stays far inside the range
    assert np.sqrt(512) < 2688


def test_packing_order_low_nibble_first():
    codes = np.array([[1, 2, 3, 4]], dtype=np.uint8)
    assert list(fp4.pack_codes(codes)[0]) == [0x21, 0x43]
    assert np.array_equal(fp4.unpack_codes(fp4.pack_codes(codes)), codes)
