"""Pins for per-position shortlists in the oracle (DynaSpec's position-aware
budget): a per-position shortlist is the same draft as a full-vocabulary
draft that is -inf off that position's list, so the oracle on the compact
form must agree with the oracle on the full-vocabulary form (whose rule is
pinned by brute force and the closed forms); a static list shared by all
positions and sequences is the stride-0 case; a bad list is reported only
at a position the left-to-right rule reaches."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle


def _full_from_compact(compact, lists, lens, V):
    """[B][K][S] compact logits and [B][K][S] lists -> [B][K][V] with -inf off the list."""
    B, K, S = compact.shape
    full = torch.full((B, K, V), -math.inf)
    for b in range(B):
        for i in range(K):
            n = lens[i]
            full[b, i, torch.as_tensor(lists[b, i, :n], dtype=torch.long)] = compact[b, i, :n]
    return full


def _case(seed, B=12, K=4, V=300, S=64):
    g = torch.Generator().manual_seed(seed)
    target = 1.5 * torch.randn((B, K + 1, V), generator=g)
    lens = [S, S, S // 2, S // 4][:K]
    lists = np.zeros((B, K, S), dtype=np.int32)
    for b in range(B):
        for i in range(K):
            lists[b, i, :lens[i]] = np.sort(torch.randperm(V, generator=g)[:lens[i]].numpy())
    compact = torch.zeros((B, K, S))
    for b in range(B):
        for i in range(K):
            idx = torch.as_tensor(lists[b, i, :lens[i]], dtype=torch.long)
            compact[b, i, :lens[i]] = target[b, i, idx] + 0.5 * torch.randn(lens[i], generator=g)
    # drafted tokens: mostly on the list, some off it (p = 0: accepted)
    tokens = np.zeros((B, K), dtype=np.int32)
    for b in range(B):
        for i in range(K):
            on = torch.rand(1, generator=g).item() < 0.9
            tokens[b, i] = lists[b, i, int(torch.randint(0, lens[i], (1,), generator=g))] if on else \
                int(torch.randint(0, V, (1,), generator=g))
    return target, compact, lists, lens, tokens


def test_per_position_lists_equal_the_full_vocabulary_form():
    for seed in range(6):
        target, compact, lists, lens, tokens = _case(seed)
        V = target.shape[-1]
        a = oracle.verify(target, compact, tokens, 0.9, 17 + seed, shortlist=lists, shortlist_len=lens, full=True)
        b = oracle.verify(target, _full_from_compact(compact, lists, lens, V), tokens, 0.9, 17 + seed, full=True)
        assert np.array_equal(a["tokens"], b["tokens"])
        assert np.array_equal(a["accept_len"], b["accept_len"])
        assert np.allclose(a["residual_mass"], b["residual_mass"], rtol=1e-12, atol=0)
        assert np.allclose(a["q_draft"], b["q_draft"], rtol=1e-12)
        assert np.allclose(a["p_draft"], b["p_draft"], rtol=1e-12)


def test_static_shared_list():
    target, compact, lists, lens, tokens = _case(11)
    B, K, S = compact.shape
    V = target.shape[-1]
    shared = lists[0, 0]                      # one list for every sequence and position
    L = np.broadcast_to(shared, (B, K, S)).copy()
    comp = torch.stack([torch.stack([target[b, i, torch.as_tensor(shared, dtype=torch.long)] for i in range(K)])
                        for b in range(B)])
    a = oracle.verify(target, comp, tokens, 1.0, 3, shortlist=shared)
    b = oracle.verify(target, _full_from_compact(comp, L, [S] * K, V), tokens, 1.0, 3)
    c = oracle.verify(target, comp, tokens, 1.0, 3, shortlist=L)
    assert np.array_equal(a["tokens"], b["tokens"]) and np.array_equal(a["tokens"], c["tokens"])


def test_bad_list_reported_only_where_reached():
    target, compact, lists, lens, tokens = _case(4, B=40)
    bad = lists.copy()
    bad[:, 2, 1] = bad[:, 2, 0]               # position 2's list is not strictly ascending
    ref = oracle.verify(target, compact, tokens, 1.0, 9, shortlist=lists, shortlist_len=lens)
    out = oracle.verify(target, compact, tokens, 1.0, 9, shortlist=bad, shortlist_len=lens)
    reach = ref["accept_len"] >= 2
    assert reach.any() and (~reach).any()
    assert (out["accept_len"][reach] == -4).all()
    assert np.array_equal(out["tokens"][~reach], ref["tokens"][~reach])
