"""FP4 main-KV format: E2M1 elements with one E4M3 scale per 16 channels.

Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression",
picx.dev summary, Methodology / Architecture Components / 5. FP4 Main KV Cache.
The page calls the format "OCP MXFP4" but gives E2M1 elements with an E4M3
scale per 16 channels and a range of 2688 = 6 * 448 (E2M1 max times E4M3 max);
that is the reading taken here (no second-level tensor scale).

Readings where the page is silent:
  * scale s = E4M3_RNE_satfinite(fl32(amax / 6)), amax = max |x| over the block
    (the choice that puts the block maximum on the largest E2M1 magnitude);
  * element code c = E2M1_RNE_satfinite(fl32(x / s)); ties go to the even code;
  * a block whose scale rounds to 0 stores all-zero codes;
  * a value rounding to magnitude 0 stores +0 (code 0), never -0;
  * packing: element 2i in the low nibble of byte i, 2i+1 in the high nibble;
    scale byte j covers elements 16j .. 16j+15.

All rounding decisions are taken on fp32 operands (as stored / as divided in
fp32), compared exactly in float64. Tables are enumerated from the format
definitions, not from any library.
"""
from __future__ import annotations

import numpy as np

BLOCK = 16

# E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; no inf/NaN.
E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E2M1_MAX = 6.0


def _e4m3_table() -> np.ndarray:
    """Values of the 256 E4M3 (OCP 'FN' variant) codes: bias 7, no inf, NaN = S.1111.111."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        s = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = s * m * 2.0 ** -9          # subnormal: (m/8) * 2^(1-7)
        else:
            vals[code] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


E4M3_VALUES = _e4m3_table()
E4M3_POS = E4M3_VALUES[:0x7F]       # codes 0x00 .. 0x7E, ascending, all finite, non-negative
E4M3_MAX = float(E4M3_POS[-1])      # 448


def e2m1_value(codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.int64)
    mag = E2M1_MAG[codes & 7]
    return np.where(codes & 8, -mag, mag)


def e4m3_value(codes) -> np.ndarray:
    return E4M3_VALUES[np.asarray(codes, dtype=np.int64)]


def _nearest_even(v: np.ndarray, mags: np.ndarray) -> np.ndarray:
    """Index into ascending `mags` of the value nearest to v >= 0 (ties -> even index).

    Values above the largest magnitude saturate to it. The index parity equals
    the code's mantissa LSB for both tables used here, so "even index" is
    "even code".
    """
    v = np.asarray(v, dtype=np.float64)
    hi = np.searchsorted(mags, v, side="left")          # first mags[hi] >= v
    hi = np.minimum(hi, len(mags) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = v - mags[lo]
    d_hi = mags[hi] - v
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(v >= mags[-1], len(mags) - 1, idx)
    idx = np.where(v <= 0.0, 0, idx)
    return idx.astype(np.int64)


def e4m3_encode_nonneg(s: np.ndarray) -> np.ndarray:
    """E4M3 code of fp32 values s >= 0, round to nearest even, saturating at 448."""
    return _nearest_even(np.asarray(s, dtype=np.float32).astype(np.float64), E4M3_POS)


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """E2M1 code of fp32 values, round to nearest even, saturating at +-6, zero as +0."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    mag_code = _nearest_even(np.abs(v), E2M1_MAG)
    neg = (v < 0) & (mag_code != 0)
    return (mag_code | np.where(neg, 8, 0)).astype(np.int64)


def quantize_blocks(x: np.ndarray):
    """Quantise fp32 rows [R, D] (D % 16 == 0) to element codes [R, D] and scale codes [R, D/16]."""
    x = np.asarray(x, dtype=np.float32)
    R, D = x.shape
    assert D % BLOCK == 0
    xb = x.reshape(R, D // BLOCK, BLOCK)
    amax = np.max(np.abs(xb), axis=2)                                   # fp32, exact
    s_f = (amax / np.float32(6.0)).astype(np.float32)                   # fl32(amax / 6)
    s_code = e4m3_encode_nonneg(s_f)
    s_val = E4M3_VALUES[s_code].astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (xb / s_val[:, :, None]).astype(np.float32)             # fl32(x / s)
    codes = e2m1_encode(ratio)
    codes = np.where((s_val == 0)[:, :, None], 0, codes)
    return codes.reshape(R, D), s_code


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """[R, D] nibbles -> [R, D/2] bytes, element 2i low nibble, 2i+1 high nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    R, Dh = packed.shape
    out = np.empty((R, 2 * Dh), dtype=np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def encode(x: np.ndarray):
    """fp32 rows [R, D] -> (packed codes uint8 [R, D/2], scale codes uint8 [R, D/16])."""
    codes, s_code = quantize_blocks(x)
    return pack_codes(codes), s_code.astype(np.uint8)


def decode(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dequantise to float64: value = e2m1(code) * e4m3(scale), exact."""
    codes = unpack_codes(packed)
    R, D = codes.shape
    vals = e2m1_value(codes).reshape(R, D // BLOCK, BLOCK)
    s = e4m3_value(np.asarray(scales, dtype=np.int64))
    return (vals * s[:, :, None]).reshape(R, D)
