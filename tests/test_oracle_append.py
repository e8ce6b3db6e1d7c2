"""Pins of the cache-append oracle against what its definition fixes, not against its
ring arithmetic: the window is the list of the last n_win tokens (brute force over a
token history), and entry e holds the FP4 encoding (pinned in test_oracle_fp4.py) of the
entry completed by token 4e+3.

Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression": blog repost
(sliding window over the most recent n_win tokens), wesearch.press card (4:1
block compression), picx.dev summary, Methodology / 5 (FP4 entries).
"""
import inspect
import types

import numpy as np
import pytest

from oracle import append, fp4


def _state(B, N, n_win, D=576):
    return dict(swa_kv=np.zeros((B, 2 * n_win, D), np.float32), kv_codes=np.full((B, N, 288), 0xAB, np.uint8),
                kv_scales=np.full((B, N, 36), 0xCD, np.uint8), z=np.full((B, N, 64), -7.0, np.float32),
                n_visible=np.full(B, -5, np.int64), win_start=np.full(B, -5, np.int64),
                win_len=np.full(B, -5, np.int64))


def _append(st, n_tokens, swa_row, entry_kv, entry_z, n_win, mod=append, **kw):
    return mod.cache_append(n_tokens, swa_row, st["swa_kv"], n_win, entry_kv, entry_z, st["kv_codes"],
                            st["kv_scales"], st["z"], st["n_visible"], st["win_start"], st["win_len"], **kw)


@pytest.mark.parametrize("n_win", [1, 2, 5, 8])
def test_window_is_the_last_n_win_tokens(n_win):
    _pin_window(append, n_win)


def _pin_window(mod, n_win):
    rng = np.random.default_rng(n_win)
    B, N = 1, 16
    st = _state(B, N, n_win, D=8)
    n_tok = np.zeros(B, np.int64)
    history = []
    for p in range(4 * n_win + 7):
        row = rng.standard_normal((B, 8)).astype(np.float32)
        history.append(row[0])
        _append(st, n_tok, row, None, None, n_win, mod)
        assert n_tok[0] == p + 1
        s, l = int(st["win_start"][0]), int(st["win_len"][0])
        want = np.array(history[max(0, len(history) - n_win):])
        assert l == len(want)
        assert np.array_equal(st["swa_kv"][0, s:s + l], want), f"window after token {p}"


def test_entries_every_fourth_token():
    _pin_entries(append)


def _pin_entries(mod):
    rng = np.random.default_rng(5)
    B, N, n_win, P = 2, 12, 4, 30
    st = _state(B, N, n_win)
    n_tok = np.zeros(B, np.int64)
    ent = rng.standard_normal((P, B, 576)).astype(np.float32)
    zz = rng.standard_normal((P, B, 64)).astype(np.float32)
    for p in range(P):
        w = _append(st, n_tok, np.zeros((B, 576), np.float32), ent[p], zz[p], n_win, mod)
        assert [e for _, e in w] == ([(p + 1) // 4 - 1] * B if (p + 1) % 4 == 0 else [])
        assert np.all(st["n_visible"] == (p + 1) // 4)
    n_e = P // 4
    for b in range(B):
        c, s = fp4.encode(ent[3::4][:n_e, b])
        assert np.array_equal(st["kv_codes"][b, :n_e], c) and np.array_equal(st["kv_scales"][b, :n_e], s)
        assert np.array_equal(st["z"][b, :n_e], zz[3::4][:n_e, b])
        # later entries untouched
        assert np.all(st["kv_codes"][b, n_e:] == 0xAB) and np.all(st["kv_scales"][b, n_e:] == 0xCD)
        assert np.all(st["z"][b, n_e:] == -7.0)


def test_ragged_positions_idle_sequences_and_no_advance():
    """Sequences at different positions (a long history replayed token by token), one idle;
    advance=False leaves n_tokens alone."""
    _pin_ragged(append)


def _pin_ragged(mod):
    rng = np.random.default_rng(6)
    n_win, N = 6, 400
    starts = [0, 3, 7, -1, 1001]
    B = len(starts)
    st = _state(B, N, n_win, D=8)
    hist = [[] for _ in range(B)]
    # build every active sequence's history up to its start position
    n_tok = np.array([0 if s >= 0 else -1 for s in starts], np.int64)
    for p in range(max(starts)):
        row = rng.standard_normal((B, 8)).astype(np.float32)
        active = np.array([0 <= n_tok[b] < starts[b] for b in range(B)])
        nt = np.where(active, n_tok, -1)
        _append(st, nt, row, None, None, n_win, mod)
        for b in range(B):
            if active[b]:
                hist[b].append(row[b])
        n_tok = np.where(active, nt, n_tok)
    assert list(n_tok) == [0, 3, 7, -1, 1001]
    before = {k: v.copy() for k, v in st.items()}
    row = rng.standard_normal((B, 8)).astype(np.float32)
    nt = n_tok.copy()
    _append(st, nt, row, None, None, n_win, mod, advance=False)
    assert np.array_equal(nt, n_tok)
    for b in range(B):
        if starts[b] < 0:
            for k in st:
                assert np.array_equal(st[k][b], before[k][b]), k
            continue
        h = hist[b] + [row[b]]
        s, l = int(st["win_start"][b]), int(st["win_len"][b])
        assert np.array_equal(st["swa_kv"][b, s:s + l], np.array(h[-n_win:]))
        assert st["n_visible"][b] == (starts[b] + 1) // 4


def test_window_after_closed_form_examples():
    _pin_closed_form(append)


def _pin_closed_form(mod):
    append = mod
    # first tokens fill the ring from row 0; from token n_win on the start walks around it
    assert append.window_after(0, 4) == (0, 1)
    assert append.window_after(3, 4) == (0, 4)
    assert append.window_after(4, 4) == (1, 4)
    assert append.window_after(7, 4) == (0, 4)
    assert append.window_after(130, 128) == (3, 128)


# Mistakes planted in a copy of the oracle (its source with one expression changed, run as
# a module of the oracle package on the CPU): each must fail at least one pin above.
MUTANTS = [
    ("ring slot", "slot = p % n_win", "slot = (p + 1) % n_win"),
    ("mirror row", "swa_kv[b, slot + n_win] = swa_row[b]", "swa_kv[b, slot] = swa_row[b]"),
    ("window length", "length = min(p + 1, n_win)", "length = min(p, n_win)"),
    ("entry index", "e = (p + 1) // ratio - 1", "e = (p + 1) // ratio"),
    ("completion rule", "if (p + 1) % ratio == 0:", "if p % ratio == 0:"),
    ("n_visible", "n_visible[b] = (p + 1) // ratio", "n_visible[b] = p // ratio"),
]


def _variant(old=None, new=None):
    src = inspect.getsource(append)
    if old is not None:
        assert src.count(old) == 1, old
        src = src.replace(old, new)
    mod = types.ModuleType("oracle._append_variant")
    mod.__package__ = "oracle"
    exec(compile(src, "<cache_append variant>", "exec"), mod.__dict__)
    return mod


def _failed_pins(mod):
    pins = [lambda w=w: _pin_window(mod, w) for w in (1, 2, 5, 8)]
    pins += [lambda: _pin_entries(mod), lambda: _pin_ragged(mod), lambda: _pin_closed_form(mod)]
    failed = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, IndexError):
            failed += 1
    return failed


def test_unchanged_copy_passes_every_pin():
    assert _failed_pins(_variant()) == 0


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(name, old, new):
    assert _failed_pins(_variant(old, new)) > 0, f"planted mistake '{name}' passes every pin"
