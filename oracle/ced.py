"""CED prefill KV projection, Eq. (1), with the FP4 cache write.

Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression",
picx.dev summary, Methodology / Architecture Components / 1. Causal
Encoder-Decoder (CED), Eq. (1): C_l = H_{L/2} W_l^KV and Z_l = H_{L/2} W_l^Z
for every decoder layer l > L/2. The wesearch.press card gives 20 of the 40
layers as the encoder, so 20 decoder layers are projected.

Readings:
  * C_l (576 channels) is the layer's main KV and is stored in the FP4 format
    of oracle.fp4, quantised from the fp32-rounded product;
  * Z_l (64 channels) is the layer's indexer key and is stored in bf16
    (round to nearest even of the exact product);
  * weights are given as W^T, one row of d_model weights per output channel.
"""
from __future__ import annotations

import numpy as np

from . import fp4


def to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned as float64.

    Written from the bf16 definition (8 significant bits, fp32 exponent range);
    finite normal inputs only.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                    # x = m * 2^e, 0.5 <= |m| < 1
    scaled = np.ldexp(m, 8)               # 8 significant bits -> integer part
    r = np.round(scaled)                  # numpy rounds half to even
    return np.ldexp(r, e - 8)


def project(Hrows: np.ndarray, W_kv_l: np.ndarray, W_z_l: np.ndarray):
    """One layer: H [R, d] (values), W_kv_l [576, d], W_z_l [64, d] -> (C float64, Z float64)."""
    Hd = np.asarray(Hrows, dtype=np.float64)
    C = Hd @ np.asarray(W_kv_l, dtype=np.float64).T
    Z = Hd @ np.asarray(W_z_l, dtype=np.float64).T
    return C, Z


def project_and_encode(Hrows, W_kv_l, W_z_l):
    """Returns (packed codes [R, 288], scales [R, 36], Z bf16 values [R, 64], C fp32 [R, 576])."""
    C, Z = project(Hrows, W_kv_l, W_z_l)
    C32 = C.astype(np.float32)
    codes, scales = fp4.encode(C32)
    return codes, scales, to_bf16_rne(Z), C32


def ambiguity_bound(Hrows, W_kv_l) -> np.ndarray:
    """Per-element bound on |fp32-accumulated product - exact product| for a length-d dot.

    gamma_d * sum_k |h_k| |w_k| with gamma_d = d u / (1 - d u), u = 2^-24: the
    classical bound for recursive summation in IEEE single precision, which
    covers any summation order.
    """
    Hd = np.abs(np.asarray(Hrows, dtype=np.float64))
    Wd = np.abs(np.asarray(W_kv_l, dtype=np.float64))
    d = Hd.shape[1]
    u = 2.0 ** -24
    gamma = d * u / (1 - d * u)
    return gamma * (Hd @ Wd.T)
