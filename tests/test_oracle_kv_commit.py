"""Pins for the KV-commit oracle: the page's rollback exercise (golden),
and invariants that a mistaken copy (wrong offset, wrong count, wrong
sequence or layer) would break."""
from __future__ import annotations

import json
import os

import numpy as np

from oracle.kv_commit import ERR_CAPACITY, kv_commit

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_rollback_exercise.json")


def _entries(tokens, W=8):
    """One distinct KV entry per token id: W bytes encoding the id."""
    return np.stack([np.full(W, t, dtype=np.uint8) for t in tokens])


def test_rollback_exercise_from_the_page():
    g = json.load(open(GOLDEN))
    P, N = g["prefix_tokens"], g["drafted_tokens"]
    L, W = 32, 8
    cache = np.zeros((1, 1, L, W), dtype=np.uint8)
    cache[0, 0, :P] = _entries(range(1, P + 1))
    staged = _entries(range(100, 100 + N))[None, None]   # the verification pass's K new entries
    accepted = g["rejected_position_1_based"] - 1
    assert accepted == g["accepted_drafts"]
    out, ln, st = kv_commit(cache, staged, [P], [accepted])
    assert ln[0] == g["cache_length_after"] and st[0] == 0
    # the next iteration reads exactly the prefix and the first accepted drafts
    expect = np.concatenate([_entries(range(1, P + 1)), _entries(range(100, 100 + accepted))])
    assert np.array_equal(out[0, 0, :ln[0]], expect)


def test_invariants_over_a_batch():
    rng = np.random.default_rng(0)
    NL, B, L, K, W = 3, 7, 40, 5, 16
    cache = rng.integers(0, 256, (NL, B, L, W), dtype=np.uint8)
    staged = rng.integers(0, 256, (NL, B, K, W), dtype=np.uint8)
    seq_len = np.array([0, 10, 35, 36, 20, 5, 40], dtype=np.int32)
    acc = np.array([3, 0, 5, 5, -2, 4, 0])     # b=3 overflows (36 + 5 > 40), b=4 is an error sequence
    out, ln, st = kv_commit(cache, staged, seq_len, acc)
    for b in range(B):
        a = acc[b]
        if a < 0:
            assert ln[b] == seq_len[b] and st[b] == 0
            assert np.array_equal(out[:, b], cache[:, b])
        elif seq_len[b] + a > L:
            assert st[b] == ERR_CAPACITY and ln[b] == seq_len[b]
            assert np.array_equal(out[:, b], cache[:, b])
        else:
            n = seq_len[b]
            assert st[b] == 0 and ln[b] == n + a
            assert np.array_equal(out[:, b, n:n + a], staged[:, b, :a])     # every layer
            assert np.array_equal(out[:, b, :n], cache[:, b, :n])           # the prefix is kept
            assert np.array_equal(out[:, b, n + a:], cache[:, b, n + a:])   # nothing past the commit


def test_in_place_commit_only_moves_the_length():
    cache = np.arange(2 * 3 * 10 * 4, dtype=np.int16).reshape(2, 3, 10, 4)
    out, ln, st = kv_commit(cache, None, [2, 5, 9], [3, 0, 2])
    assert np.array_equal(out, cache)
    assert ln.tolist() == [5, 5, 9] and st.tolist() == [0, 0, ERR_CAPACITY]
