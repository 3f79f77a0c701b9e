"""Pins for the oracle outputs that the GPU parity checks lean on.

The GPU's per-position outputs are held to the oracle's q_i(d_i), p_i(d_i) and
per-row log-sum-exp, and GPU/oracle token differences are excused only where
the oracle's accept or sample margin is below 1e-6.  Each of those outputs is
checked here against something outside the oracle: scipy's logsumexp and
softmax, the printed five-word example of the runelab.ai post (§ the exact
rule), the Philox words rebuilt into uniforms with the rule min(1, q/p)
evaluated by numpy, and numpy.searchsorted on the normalised CDF.

Every test names, in its docstring, the one-line mistakes in oracle.c that it
was seen to catch (each planted in the oracle on the CPU, the suite run, the
mistake taken out again).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _case(B, K, V, T, seed, dtype=torch.float32, sigma=0.7):
    """Random logits with a few -inf entries; draft = target + noise; drafted
    tokens from the draft softmax (numpy's sampler)."""
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 2.0, size=(B, K + 1, V))
    zd = zt[:, :K] + rng.normal(0, sigma, size=(B, K, V))
    zt[rng.random(zt.shape) < 0.03] = -np.inf
    zd[rng.random(zd.shape) < 0.03] = -np.inf
    tgt = torch.tensor(zt, dtype=torch.float32).to(dtype)
    drf = torch.tensor(zd, dtype=torch.float32).to(dtype)
    zd64 = drf.double().numpy()
    tok = np.zeros((B, K), dtype=np.int32)
    for b in range(B):
        for i in range(K):
            tok[b, i] = rng.choice(V, p=softmax(zd64[b, i] / T))
    return tgt, drf, tok


def _key(seed):
    return [seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF]


def _uniform(seed, b, pos, word):
    """The verification uniform, rebuilt from the Philox word as (n + 1/2) 2^-24."""
    w = int(oracle.philox4x32_10([pos, b, 0, 0], _key(seed))[word])
    return ((w >> 8) + 0.5) / 2.0 ** 24


@pytest.mark.parametrize("T,dtype", [(0.7, torch.float32), (1.3, torch.float32), (1.0, torch.bfloat16)])
def test_row_lse_is_scipy_logsumexp(T, dtype):
    """row_lse[b][i] = logsumexp(z / T) of target row i (slots 0..K) and draft
    row i (slots K+1..2K), by scipy.special.logsumexp.

    Caught mistakes: the log-sum-exp returned as zmax + log(sum) without the
    division by T; a draft row's value written to slot i instead of K+1+i."""
    B, K, V = 7, 3, 61
    tgt, drf, tok = _case(B, K, V, T, seed=int(T * 10))
    tgt, drf = tgt.to(dtype), drf.to(dtype)
    out = oracle.verify(tgt, drf, tok, T, seed=5, full=True)
    zt, zd = tgt.double().numpy(), drf.double().numpy()
    want = np.concatenate([logsumexp(zt / T, axis=-1), logsumexp(zd / T, axis=-1)], axis=1)
    np.testing.assert_allclose(out["row_lse"], want, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("T", [0.6, 1.0, 1.7])
def test_q_and_p_at_drafted_token_are_numpy_softmax(T):
    """q_draft[b][i] = softmax(zt_i / T)[d_i] and p_draft[b][i] = softmax(zd_i / T)[d_i]
    for every position, examined or not, by scipy.special.softmax.

    Caught mistakes: q and p swapped; the drafted token's neighbour d + 1 read;
    the draft row's temperature left out."""
    B, K, V = 9, 4, 47
    tgt, drf, tok = _case(B, K, V, T, seed=3)
    out = oracle.verify(tgt, drf, tok, T, seed=11, full=True)
    zt, zd = tgt.double().numpy(), drf.double().numpy()
    qd = np.take_along_axis(softmax(zt[:, :K] / T, axis=-1), tok[..., None].astype(np.int64), -1)[..., 0]
    pd = np.take_along_axis(softmax(zd / T, axis=-1), tok[..., None].astype(np.int64), -1)[..., 0]
    np.testing.assert_allclose(out["q_draft"], qd, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(out["p_draft"], pd, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("probs", [False, True])
def test_q_and_p_five_word_example(probs):
    """The runelab.ai single-position figure (§ the exact rule): target
    42/26/16/10/6 %, draft 20/45/10/5/20 %.  Drafting word w returns
    q(w) and p(w) as printed (first word: 42 % and 20 %), from logits ln q,
    ln p stored in float32, or from the printed draft probabilities.

    Caught mistakes: q and p swapped; the drafted token's neighbour read."""
    g = json.load(open(os.path.join(GOLDEN, "worked_example_five_words.json")))
    q = np.array(g["target_percent"], dtype=np.float64) / 100
    p = np.array(g["draft_percent"], dtype=np.float64) / 100
    B, K, V = 5, 1, 5
    tgt = torch.tensor(np.log(q), dtype=torch.float32).expand(B, K + 1, V).contiguous()
    if probs:
        drf = torch.tensor(p, dtype=torch.float32).expand(B, K, V).contiguous()
    else:
        drf = torch.tensor(np.log(p), dtype=torch.float32).expand(B, K, V).contiguous()
    tok = np.arange(B, dtype=np.int32).reshape(B, K)
    out = oracle.verify(tgt, drf, tok, 1.0, seed=1, full=True, draft_is_probs=probs)
    np.testing.assert_allclose(out["q_draft"][:, 0], q, rtol=0, atol=2e-7)
    np.testing.assert_allclose(out["p_draft"][:, 0], p, rtol=0, atol=2e-7)
    assert abs(out["q_draft"][0, 0] - 0.42) < 2e-7 and abs(out["p_draft"][0, 0] - 0.20) < 2e-7


def test_accept_margin_is_distance_to_min_one_ratio():
    """accept_margin[b][i] = |u_i - min(1, q_i(d_i) / p_i(d_i))| at every
    position the left-to-right rule examines (u_i rebuilt from Philox word 0
    of counter (i, b, 0, 0)), and +inf elsewhere and where p_i(d_i) = 0; the
    accept decisions are u_i < min(1, q/p).

    Caught mistakes: the margin written without the absolute value; measured
    to q/p instead of min(1, q/p); stored at position i + 1."""
    B, K, V, T, seed = 160, 4, 40, 0.8, 0x1234_5678_9ABC
    tgt, drf, tok = _case(B, K, V, T, seed=17, sigma=0.6)
    # a few drafted tokens the draft gives probability 0: accepted, no margin
    drf = drf.clone()
    for b in (3, 50, 99):
        drf[b, 0, int(tok[b, 0])] = -math.inf
    out = oracle.verify(tgt, drf, tok, T, seed=seed)
    zt, zd = tgt.double().numpy(), drf.double().numpy()
    seen_ratio_above_one = seen_reject = 0
    for b in range(B):
        L = int(out["accept_len"][b])
        assert 0 <= L <= K
        for i in range(K):
            m = out["accept_margin"][b, i]
            if i > L or (i == L and L == K):
                assert m == math.inf, (b, i)
                continue
            qd = softmax(zt[b, i] / T)[tok[b, i]]
            pd = softmax(zd[b, i] / T)[tok[b, i]]
            u = _uniform(seed, b, i, 0)
            if pd == 0.0:
                assert m == math.inf and i < L, (b, i)
                continue
            a = min(1.0, qd / pd)
            seen_ratio_above_one += qd > pd
            assert abs(m - abs(u - a)) < 1e-12, (b, i, m, u, a)
            assert (u < a) == (i < L), (b, i)
            seen_reject += i == L
    assert seen_ratio_above_one > 20 and seen_reject > 20


def test_sample_margin_and_residual_mass_by_searchsorted():
    """At the end position j the emitted token is numpy.searchsorted of the
    uniform v (Philox word 1 of counter (j, b, 0, 0)) in the normalised CDF
    of r = max(0, q_j - p_j) (q_K for the bonus); sample_margin is v's
    distance to the nearer edge of that token's interval [C(x-1), C(x)), and
    residual_mass is sum r.

    Caught mistakes: the margin measured to the upper edge only; to the lower
    edge only; the CDF not divided by R."""
    B, K, V, T, seed = 200, 3, 33, 1.1, 77
    tgt, drf, tok = _case(B, K, V, T, seed=23, sigma=0.9)
    out = oracle.verify(tgt, drf, tok, T, seed=seed)
    zt, zd = tgt.double().numpy(), drf.double().numpy()
    lower_nearer = upper_nearer = 0
    for b in range(B):
        j = int(out["accept_len"][b])
        q = softmax(zt[b, j] / T)
        r = q if j == K else np.maximum(0.0, q - softmax(zd[b, j] / T))
        R = r.sum()
        if j < K:
            assert abs(out["residual_mass"][b] - R) < 1e-12
        C = np.cumsum(r) / R
        v = _uniform(seed, b, j, 1)
        x = int(np.searchsorted(C, v, side="right"))
        assert out["tokens"][b, j] == x, b
        lo = v - (C[x - 1] if x > 0 else 0.0)
        hi = C[x] - v
        assert abs(out["sample_margin"][b] - min(lo, hi)) < 1e-12, b
        lower_nearer += lo < hi
        upper_nearer += hi < lo
    assert lower_nearer > 20 and upper_nearer > 20


def test_draws_with_given_probabilities_by_numpy():
    """With draft probabilities given, the accept decisions are u_i <
    min(1, q_i(d_i) / p_i(d_i)) with p read as given (no softmax, no T), and
    the emitted token is numpy.searchsorted of v in the normalised CDF of
    max(0, q_j - p_j) (q_K for the bonus); residual_mass is its total.

    Caught mistakes the logit pins cannot: the temperature applied to the given
    probabilities, or their logarithm taken as logits."""
    B, K, V, T, seed = 160, 3, 29, 0.9, 4242
    tgt, drf, tok = _case(B, K, V, T, seed=31, sigma=0.8)
    zd = drf.double().numpy()
    probs = np.stack([[softmax(zd[b, i]) for i in range(K)] for b in range(B)])   # not the T-softmax
    out = oracle.verify(tgt, torch.tensor(probs, dtype=torch.float32), tok, T, seed=seed, draft_is_probs=True)
    p32 = torch.tensor(probs, dtype=torch.float32).double().numpy()   # the values the oracle was given
    zt = tgt.double().numpy()
    n_rej = n_bonus = 0
    for b in range(B):
        L = K
        for i in range(K):
            q = softmax(zt[b, i] / T)
            pd = p32[b, i, tok[b, i]]
            acc = pd == 0.0 or _uniform(seed, b, i, 0) < min(1.0, q[tok[b, i]] / pd)
            if not acc:
                L = i
                break
        assert int(out["accept_len"][b]) == L, b
        q = softmax(zt[b, L] / T)
        r = q if L == K else np.maximum(0.0, q - p32[b, L])
        R = r.sum()
        if L < K:
            assert abs(out["residual_mass"][b] - R) < 1e-12, b
            n_rej += 1
        else:
            n_bonus += 1
        x = int(np.searchsorted(np.cumsum(r) / R, _uniform(seed, b, L, 1), side="right"))
        assert out["tokens"][b, L] == x, b
        assert list(out["tokens"][b, :L]) == list(tok[b, :L]), b
    assert n_rej > 20 and n_bonus > 5


def test_draws_with_a_shortlisted_draft_by_numpy():
    """With a shortlisted draft (compact logits over a per-sequence list), p_i
    is the softmax of the listed logits at T placed on the listed tokens and 0
    elsewhere; the accept decisions are u_i < min(1, q_i(d_i) / p_i(d_i))
    (always when p_i(d_i) = 0) and the emitted token is numpy.searchsorted of v
    in the normalised CDF of max(0, q_j - p_j) over the full vocabulary.

    Caught mistakes: the list's logits scattered one token off; the residual
    taken over the listed tokens only."""
    B, K, V, S, T, seed = 120, 3, 37, 12, 0.8, 99
    rng = np.random.default_rng(5)
    zt = rng.normal(0, 2.0, size=(B, K + 1, V))
    lists = np.stack([np.sort(rng.choice(V, size=S, replace=False)) for _ in range(B)]).astype(np.int32)
    zd = np.stack([zt[b, :K][:, lists[b]] for b in range(B)]) + rng.normal(0, 0.7, size=(B, K, S))
    tok = np.zeros((B, K), dtype=np.int32)
    for b in range(B):
        for i in range(K):
            # mostly listed tokens, now and then one off the list (p = 0: accepted)
            tok[b, i] = lists[b][rng.choice(S, p=softmax(zd[b, i] / T))] if rng.random() > 0.05 else rng.integers(V)
    tgt = torch.tensor(zt, dtype=torch.float32)
    drf = torch.tensor(zd, dtype=torch.float32)
    out = oracle.verify(tgt, drf, tok, T, seed=seed, shortlist=torch.tensor(lists))
    zt32, zd32 = tgt.double().numpy(), drf.double().numpy()
    n_rej = n_off = 0
    for b in range(B):
        p = np.zeros((K, V))
        for i in range(K):
            p[i, lists[b]] = softmax(zd32[b, i] / T)
        L = K
        for i in range(K):
            q = softmax(zt32[b, i] / T)
            pd = p[i, tok[b, i]]
            n_off += pd == 0.0
            if not (pd == 0.0 or _uniform(seed, b, i, 0) < min(1.0, q[tok[b, i]] / pd)):
                L = i
                break
        assert int(out["accept_len"][b]) == L, b
        q = softmax(zt32[b, L] / T)
        r = q if L == K else np.maximum(0.0, q - p[L])
        n_rej += L < K
        x = int(np.searchsorted(np.cumsum(r) / r.sum(), _uniform(seed, b, L, 1), side="right"))
        assert out["tokens"][b, L] == x, b
    assert n_rej > 20 and n_off > 3
