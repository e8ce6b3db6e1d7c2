"""Decode-time cache append: one new token per sequence.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression":
  * blog repost (zartbot essay), introduction: the sliding-window branch covers the
    local window, the most recent n_win tokens;
  * wesearch.press card: block-based compression shrinks the KV cache by a factor of
    four (four tokens per compressed entry);
  * picx.dev summary, Methodology / 5. FP4 Main KV Cache: the compressed entries are
    stored as E2M1 codes with one E4M3 scale per 16 channels (fp4.encode).

Readings where the pages are silent:
  * the window after appending token p (0-based) holds tokens max(0, p+1-n_win) .. p,
    the new token included;
  * token p completes compressed entry e = (p+1)/ratio - 1 when (p+1) % ratio == 0
    (ratio = 4); how tokens are compressed into an entry is not described, so the
    entry's latent row and indexer key are inputs; the entry is visible from that
    token on: n_visible = (p+1) // ratio;
  * the window rows live in a mirrored ring of R = n_win slots stored twice
    (rows 0..2R-1): token p goes to rows p % R and p % R + R, so the window is the
    contiguous run of rows starting at (p+1-len) % R, len = min(p+1, n_win), which
    the attention calls read as [win_start, win_start + win_len);
  * a sequence with n_tokens < 0 is idle: nothing is written for it.
"""
from __future__ import annotations

import numpy as np

from . import fp4

RATIO = 4


def window_after(p: int, n_win: int):
    """(win_start, win_len) of the ring window once token p is stored."""
    length = min(p + 1, n_win)
    return (p + 1 - length) % n_win, length


def cache_append(n_tokens, swa_row, swa_kv, n_win, entry_kv, entry_z, kv_codes, kv_scales, z,
                 n_visible, win_start, win_len, ratio=RATIO, advance=True):
    """Append token n_tokens[b] of every active sequence b, in place.

    n_tokens int [B]; swa_row [B, 576] (window row of the new token, any float type,
    copied as is) or None; swa_kv [B, >= 2*n_win, 576]; entry_kv float [B, 576] (the
    compressed entry the token completes) or None; entry_z [B, 64] or None; kv_codes
    uint8 [B, N, 288]; kv_scales uint8 [B, N, 36]; z [B, N, 64]; n_visible, win_start,
    win_len int [B] (outputs, may be None). Returns the list of (b, e) entries written.
    """
    written = []
    for b in range(len(n_tokens)):
        p = int(n_tokens[b])
        if p < 0:
            continue
        if swa_row is not None:
            slot = p % n_win
            swa_kv[b, slot] = swa_row[b]
            swa_kv[b, slot + n_win] = swa_row[b]
        if (p + 1) % ratio == 0:
            e = (p + 1) // ratio - 1
            if entry_kv is not None:
                c, s = fp4.encode(np.asarray(entry_kv[b], dtype=np.float32)[None, :])
                kv_codes[b, e] = c[0]
                kv_scales[b, e] = s[0]
            if entry_z is not None:
                z[b, e] = entry_z[b]
            written.append((b, e))
        if n_visible is not None:
            n_visible[b] = (p + 1) // ratio
        if win_start is not None:
            win_start[b], win_len[b] = window_after(p, n_win)
        if advance:
            n_tokens[b] = p + 1
    return written
