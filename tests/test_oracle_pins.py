"""Pins for the float64 oracle: what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: numbers the
pages print, the distribution-preservation theorem, closed forms, brute-force
enumeration, a library routine, or another implementation of Philox.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import brute
import oracle
from speculative_decoding_verification_sampling_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np_softmax(z, T=1.0):
    z = np.asarray(z, dtype=np.float64) / T
    m = np.max(z[np.isfinite(z)])
    e = np.where(np.isfinite(z), np.exp(z - m), 0.0)
    return e / e.sum()


def _sample(prob, n, rng):
    """n draws from a probability vector (numpy's own sampler)."""
    return rng.choice(len(prob), size=n, p=np.asarray(prob, dtype=np.float64) / np.sum(prob))


def _batch(q_rows, draft_rows, tokens, probs=False):
    """Replicate one set of rows over B sequences: target logits float32 ln(q)
    and draft float32 probabilities (or logits)."""
    B = tokens.shape[0]
    q = np.stack(q_rows)
    logq = np.full(q.shape, -np.inf)
    logq[q > 0] = np.log(q[q > 0])
    tgt = torch.tensor(logq, dtype=torch.float32).unsqueeze(0).expand(B, -1, -1).contiguous()
    d = torch.tensor(np.stack(draft_rows), dtype=torch.float32).unsqueeze(0).expand(B, -1, -1).contiguous()
    return tgt, d


# ------------------------------------------------------------------ Philox
_TRITON_PHILOX = r"""
import json, sys
import numpy as np, torch
import triton, triton.language as tl

@triton.jit
def kern(c_ptr, k_ptr, o_ptr, N: tl.constexpr):
    i = tl.arange(0, N)
    c0 = tl.load(c_ptr + i * 4 + 0).to(tl.uint32, bitcast=True)
    c1 = tl.load(c_ptr + i * 4 + 1).to(tl.uint32, bitcast=True)
    c2 = tl.load(c_ptr + i * 4 + 2).to(tl.uint32, bitcast=True)
    c3 = tl.load(c_ptr + i * 4 + 3).to(tl.uint32, bitcast=True)
    k0 = tl.load(k_ptr + i * 2 + 0).to(tl.uint32, bitcast=True)
    k1 = tl.load(k_ptr + i * 2 + 1).to(tl.uint32, bitcast=True)
    a, b, c, d = tl.philox_impl(c0, c1, c2, c3, k0, k1, 10)
    tl.store(o_ptr + i * 4 + 0, a.to(tl.int32, bitcast=True))
    tl.store(o_ptr + i * 4 + 1, b.to(tl.int32, bitcast=True))
    tl.store(o_ptr + i * 4 + 2, c.to(tl.int32, bitcast=True))
    tl.store(o_ptr + i * 4 + 3, d.to(tl.int32, bitcast=True))

data = json.loads(sys.stdin.read())
ctr = np.array(data["ctr"], dtype=np.uint32)
key = np.array(data["key"], dtype=np.uint32)
N = ctr.shape[0]
o = torch.zeros(N * 4, dtype=torch.int32)
kern[(1,)](torch.from_numpy(ctr.view(np.int32).reshape(-1).copy()),
           torch.from_numpy(key.view(np.int32).reshape(-1).copy()), o, N=N)
print(json.dumps(o.numpy().view(np.uint32).reshape(N, 4).tolist()))
"""


def test_philox_matches_triton_interpreter():
    """Philox4x32-10 against Triton's independent implementation (run by its
    CPU interpreter in a child process) on random counters and keys."""
    import json as _json
    import subprocess
    import sys
    pytest.importorskip("triton")
    rng = np.random.default_rng(7)
    N = 64
    ctr = rng.integers(0, 2**32, size=(N, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2**32, size=(N, 2), dtype=np.uint64).astype(np.uint32)
    ctr[0] = 0
    key[0] = 0
    ctr[1] = 0xFFFFFFFF
    key[1] = 0xFFFFFFFF
    env = dict(os.environ, TRITON_INTERPRET="1")
    res = subprocess.run([sys.executable, "-c", _TRITON_PHILOX], input=_json.dumps(
        {"ctr": ctr.tolist(), "key": key.tolist()}), capture_output=True, text=True, env=env,
        timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    want = np.array(_json.loads(res.stdout.strip().splitlines()[-1]), dtype=np.uint32)
    got = np.stack([oracle.philox4x32_10(ctr[n], key[n]) for n in range(N)])
    np.testing.assert_array_equal(got, want)


def test_uniform24_range():
    """(n + 1/2) 2^-24 with n = w >> 8: the odd multiples of 2^-25 in (0, 1),
    exact in float64.  A float32 holds it only for n < 2^23 (it needs 25
    significant bits above that)."""
    assert oracle.uniform24(0) == 2.0 ** -25
    assert oracle.uniform24(0xFFFFFFFF) == 1.0 - 2.0 ** -25
    assert np.float32(oracle.uniform24(0x12345678)) == oracle.uniform24(0x12345678)
    for w in (0x80000000, 0x80000100, 0xC0FFEE00, 0xFFFFFF00):
        u = oracle.uniform24(w)
        n = w >> 8
        assert n >= 2 ** 23
        assert u * 2.0 ** 25 == 2 * n + 1                # exact in float64
        assert float(np.float32(u)) != u                 # one bit too many for float32


# ------------------------------------------------------------------ worked example
def test_worked_example_five_words():
    """runelab.ai single-position example: 42/26/16/10/6 vs 20/45/10/5/20
    accepts 67 % of drafts; the replacements are 22/0/6/5/0 (total 33)."""
    g = json.load(open(os.path.join(GOLDEN, "worked_example_five_words.json")))
    q = np.array(g["target_percent"], dtype=np.float64) / 100
    p = np.array(g["draft_percent"], dtype=np.float64) / 100
    qs, _ = oracle.softmax(np.log(q))
    np.testing.assert_allclose(qs, q, rtol=0, atol=1e-12)
    accept = sum(p[d] * oracle.accept_prob(q[d], p[d]) for d in range(5))
    assert abs(accept - g["accept_percent"] / 100) < 1e-12
    r, R = oracle.residual(q, p)
    np.testing.assert_allclose(r, np.array(g["residual_percent"]) / 100, rtol=0, atol=1e-12)
    assert abs(R - g["residual_total_percent"] / 100) < 1e-12
    # the page's split of the first two words: accepted-draft part + replacement part
    reject = sum(p[d] * (1 - oracle.accept_prob(q[d], p[d])) for d in range(5))
    for w, key in ((0, "first_word_split_percent"), (1, "second_word_split_percent")):
        accepted = p[w] * oracle.accept_prob(q[w], p[w])
        replaced = reject * r[w] / R
        assert abs(accepted - g[key]["accepted"] / 100) < 1e-12
        assert abs(replaced - g[key]["replacement"] / 100) < 1e-12


def test_worked_example_end_to_end_histogram():
    """Draws through the whole oracle round (K=1, V=5, draft probabilities as
    printed): the emitted token follows the target's 42/26/16/10/6."""
    from scipy.stats import chisquare
    g = json.load(open(os.path.join(GOLDEN, "worked_example_five_words.json")))
    q = np.array(g["target_percent"], dtype=np.float64) / 100
    p = np.array(g["draft_percent"], dtype=np.float64) / 100
    B = 100_000
    rng = np.random.default_rng(11)
    d = _sample(p, B, rng).reshape(B, 1)
    tgt, drf = _batch([q, q], [p], d)
    out = oracle.verify(tgt, drf, d, 1.0, seed=123, draft_is_probs=True)
    first = out["tokens"][:, 0]
    counts = np.bincount(first, minlength=5)
    assert chisquare(counts, q * B).pvalue > 1e-3
    acc = np.mean(out["accept_len"] == 1)
    assert abs(acc - 0.67) < 4 * math.sqrt(0.67 * 0.33 / B)


# ------------------------------------------------------------------ brute force
def _rational_case(V, K, seed):
    rng = np.random.default_rng(seed)
    q = []
    p = []
    for i in range(K + 1):
        w = rng.integers(1, 9, size=V)
        if i == 1:
            w[rng.integers(0, V)] = 0     # a zero target probability somewhere
        q.append([Fraction(int(x), int(w.sum())) for x in w])
    for i in range(K):
        w = rng.integers(0, 9, size=V)
        w[rng.integers(0, V)] += 1
        tot = int(w.sum())
        # dyadic draft probabilities so that float32 holds them exactly
        scale = 64
        raw = [int(round(int(x) * scale / tot)) for x in w]
        raw[int(np.argmax(raw))] += scale - sum(raw)
        p.append([Fraction(x, scale) for x in raw])
    return q, p


@pytest.mark.parametrize("V,K,seed", [(2, 1, 0), (3, 2, 1), (4, 2, 2), (4, 1, 3), (3, 1, 4)])
def test_brute_force_theorem(V, K, seed):
    """The enumerator reproduces the target exactly: first token ~ q_1, and
    after an accepted prefix the next token ~ q at that position."""
    q, p = _rational_case(V, K, seed)
    dist = brute.round_distribution(q, p)
    assert sum(dist.values()) == 1
    assert brute.first_token_marginal(dist, V) == q[0]
    for x in range(V):
        cond = brute.next_token_conditional(dist, (x,), V)
        if cond is not None and K >= 1:
            assert cond == q[1]


@pytest.mark.parametrize("V,K,seed", [(2, 1, 0), (3, 2, 1), (4, 2, 2), (4, 1, 3)])
def test_oracle_matches_brute_force(V, K, seed):
    """For every fixed draft-token tuple, the oracle's emitted sequences over
    many seeds follow the exact enumerated distribution (chi-square)."""
    from itertools import product
    from scipy.stats import chisquare
    q, p = _rational_case(V, K, seed)
    qf = [np.array([float(x) for x in row]) for row in q]
    pf = [np.array([float(x) for x in row]) for row in p]
    n_per = 40_000
    combos = [c for c in product(range(V), repeat=K)]
    tokens = np.repeat(np.array(combos, dtype=np.int32), n_per, axis=0)
    tgt, drf = _batch(qf, pf, tokens)
    out = oracle.verify(tgt, drf, tokens, 1.0, seed=1000 + seed, draft_is_probs=True)
    pvals = []
    for c_i, combo in enumerate(combos):
        exact = brute.round_given_drafts(q, p, combo)
        sl = slice(c_i * n_per, (c_i + 1) * n_per)
        toks, lens = out["tokens"][sl], out["accept_len"][sl]
        seen = {}
        for t_row, L in zip(toks, lens):
            key = tuple(int(x) for x in t_row[:L + 1])
            seen[key] = seen.get(key, 0) + 1
        for key in seen:
            assert key in exact, f"impossible outcome {key} for drafts {combo}"
        keys = sorted(exact)
        obs = np.array([seen.get(k, 0) for k in keys], dtype=np.float64)
        exp = np.array([float(exact[k]) for k in keys]) * n_per
        if len(keys) > 1:
            pvals.append(chisquare(obs, exp).pvalue)
    assert min(pvals) > 1e-3 / len(pvals)


# ------------------------------------------------------------------ chi-square / TV on V=8
@pytest.mark.parametrize("seed", [0, 1, 2, 3, 4])
def test_chi_square_v8(seed):
    """nextadmin.net exercise 1: the speculative histogram matches direct
    target sampling (chi-square, p > 0.05 over 50,000 tokens); five fixed
    seeds, Bonferroni threshold 0.01."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(100 + seed)
    V, K, B = 8, 3, 50_000
    zt = rng.normal(0, 1.5, size=(K + 1, V))
    zd = zt[:K] + rng.normal(0, 0.8, size=(K, V))
    T = 0.9
    p = [_np_softmax(zd[i], T) for i in range(K)]
    q1 = _np_softmax(zt[0], T)
    tokens = np.stack([_sample(p[i], B, rng) for i in range(K)], axis=1).astype(np.int32)
    tgt = torch.tensor(zt, dtype=torch.float32).unsqueeze(0).expand(B, -1, -1).contiguous()
    drf = torch.tensor(zd, dtype=torch.float32).unsqueeze(0).expand(B, -1, -1).contiguous()
    out = oracle.verify(tgt, drf, tokens, T, seed=seed)
    counts = np.bincount(out["tokens"][:, 0], minlength=V)
    assert chisquare(counts, q1 * B).pvalue > 0.01


def test_total_variation_below_001():
    """aiengineeringfromscratch.com exercise: TV distance between speculative
    output and plain target sampling below 0.01 (first and second token)."""
    rng = np.random.default_rng(5)
    V, K, B = 8, 2, 200_000
    zt = rng.normal(0, 2.0, size=(K + 1, V))
    zd = zt[:K] + rng.normal(0, 1.0, size=(K, V))
    p = [_np_softmax(zd[i]) for i in range(K)]
    tokens = np.stack([_sample(p[i], B, rng) for i in range(K)], axis=1).astype(np.int32)
    tgt = torch.tensor(zt, dtype=torch.float32).unsqueeze(0).expand(B, -1, -1).contiguous()
    drf = torch.tensor(zd, dtype=torch.float32).unsqueeze(0).expand(B, -1, -1).contiguous()
    out = oracle.verify(tgt, drf, tokens, 1.0, seed=99)
    emp1 = np.bincount(out["tokens"][:, 0], minlength=V) / B
    tv1 = 0.5 * np.abs(emp1 - _np_softmax(zt[0])).sum()
    assert tv1 < 0.01
    two = out["accept_len"] >= 1
    emp2 = np.bincount(out["tokens"][two, 1], minlength=V) / two.sum()
    tv2 = 0.5 * np.abs(emp2 - _np_softmax(zt[1])).sum()
    assert tv2 < 0.01


# ------------------------------------------------------------------ closed forms
@pytest.mark.parametrize("alpha,K", [(0.8, 4), (0.5, 3), (0.9, 6)])
def test_expected_tokens_closed_form(alpha, K):
    """E[tokens per round] = (1 - alpha^(K+1)) / (1 - alpha) for drafts whose
    per-position acceptance is exactly alpha (aiengineeringfromscratch.com
    'expected speedup': 3.36 at alpha = 0.8, K = 4)."""
    if (alpha, K) == (0.8, 4):
        assert round((1 - alpha ** (K + 1)) / (1 - alpha), 2) == 3.36
    V, B = 16, 200_000
    gen = torch.Generator().manual_seed(int(alpha * 100) + K)
    rng = np.random.default_rng(K)
    qs, ps = [], []
    for _ in range(K + 1):
        q, p = synth.controlled_alpha_pair(V, alpha, gen)
        qs.append(q.numpy())
        ps.append(p.numpy())
    tokens = np.stack([_sample(ps[i], B, rng) for i in range(K)], axis=1).astype(np.int32)
    tgt = torch.tensor(np.log(np.maximum(np.stack(qs), 1e-300)), dtype=torch.float32)
    tgt = torch.where(torch.tensor(np.stack(qs)) > 0, tgt, torch.tensor(-math.inf))
    tgt = tgt.unsqueeze(0).expand(B, -1, -1).contiguous()
    drf = torch.tensor(np.stack(ps[:K]), dtype=torch.float32).unsqueeze(0).expand(B, -1, -1).contiguous()
    out = oracle.verify(tgt, drf, tokens, 1.0, seed=4242, draft_is_probs=True)
    emitted = out["accept_len"] + 1
    expect = (1 - alpha ** (K + 1)) / (1 - alpha)
    sd = emitted.std()
    assert abs(emitted.mean() - expect) < 4 * sd / math.sqrt(B)


def test_expected_tokens_general_product_form():
    """E[tokens] = sum_k prod_{i<=k} beta_i with beta_i = sum_x min(p_i, q_i),
    on random logits (betas from numpy, independent of the oracle)."""
    rng = np.random.default_rng(21)
    V, K, B = 12, 4, 200_000
    zt = rng.normal(0, 2.0, size=(K + 1, V))
    zd = zt[:K] + rng.normal(0, 1.2, size=(K, V))
    q = [_np_softmax(zt[i]) for i in range(K + 1)]
    p = [_np_softmax(zd[i]) for i in range(K)]
    beta = [np.minimum(p[i], q[i]).sum() for i in range(K)]
    expect = sum(np.prod(beta[:k]) for k in range(K + 1))
    tokens = np.stack([_sample(p[i], B, rng) for i in range(K)], axis=1).astype(np.int32)
    tgt = torch.tensor(zt, dtype=torch.float32).unsqueeze(0).expand(B, -1, -1).contiguous()
    drf = torch.tensor(zd, dtype=torch.float32).unsqueeze(0).expand(B, -1, -1).contiguous()
    out = oracle.verify(tgt, drf, tokens, 1.0, seed=77)
    emitted = out["accept_len"] + 1
    assert abs(emitted.mean() - expect) < 4 * emitted.std() / math.sqrt(B)


# ------------------------------------------------------------------ special cases
def test_p_equals_q_always_accepts_and_bonus_is_searchsorted():
    """p == q: every draft is accepted and the bonus is inverse-CDF sampling of
    q_{K+1}, i.e. numpy.searchsorted on its cumulative sum."""
    rng = np.random.default_rng(3)
    B, K, V = 64, 3, 50
    z = torch.tensor(rng.normal(0, 2, size=(B, K + 1, V)), dtype=torch.float32)
    d = torch.tensor(np.stack([rng.integers(0, V, size=K) for _ in range(B)]), dtype=torch.int32)
    out = oracle.verify(z, z[:, :K].clone(), d, 1.0, seed=5)
    assert (out["accept_len"] == K).all()
    assert (out["tokens"][:, :K] == d.numpy()).all()
    for b in range(B):
        qK = _np_softmax(z[b, K].double().numpy())
        w = oracle.philox4x32_10([K, b, 0, 0], [5, 0])
        v = oracle.uniform24(int(w[1]))
        c = np.cumsum(qK)
        want = int(np.searchsorted(c, v * c[-1], side="right"))
        assert out["tokens"][b, K] == want


def test_one_hot_target_is_deterministic():
    B, K, V = 32, 4, 10
    rng = np.random.default_rng(8)
    t = rng.integers(0, V)
    zt = torch.full((B, K + 1, V), -math.inf)
    zt[:, :, t] = 0.0
    zd = torch.tensor(rng.normal(0, 1, size=(B, K, V)), dtype=torch.float32)
    d = torch.tensor(rng.integers(0, V, size=(B, K)), dtype=torch.int32)
    d[:B // 2, :2] = t
    out = oracle.verify(zt, zd, d, 1.0, seed=9)
    for b in range(B):
        j = 0
        while j < K and d[b, j] == t:
            j += 1
        assert out["accept_len"][b] == j
        assert list(out["tokens"][b, :j + 1]) == [t] * (j + 1)


def test_one_hot_draft_accepts_with_q_and_renormalises():
    """Draft puts all mass on d: accept with probability q(d); a replacement
    follows q with d removed, renormalised."""
    from scipy.stats import chisquare
    B, V, d = 200_000, 6, 2
    rng = np.random.default_rng(12)
    zt = rng.normal(0, 1, size=(2, V))
    q = _np_softmax(zt[0])
    zd = np.full((1, V), -math.inf)
    zd[0, d] = 0.0
    tgt = torch.tensor(zt, dtype=torch.float32).unsqueeze(0).expand(B, -1, -1).contiguous()
    drf = torch.tensor(zd, dtype=torch.float32).unsqueeze(0).expand(B, -1, -1).contiguous()
    tok = torch.full((B, 1), d, dtype=torch.int32)
    out = oracle.verify(tgt, drf, tok, 1.0, seed=31)
    acc = out["accept_len"] == 1
    assert abs(acc.mean() - q[d]) < 4 * math.sqrt(q[d] * (1 - q[d]) / B)
    rep = out["tokens"][~acc, 0]
    assert not (rep == d).any()
    want = q.copy()
    want[d] = 0
    want /= want.sum()
    counts = np.bincount(rep, minlength=V)
    keep = want > 0
    assert chisquare(counts[keep], want[keep] * len(rep)).pvalue > 1e-3


def test_greedy_matches_numpy_argmax_with_ties():
    rng = np.random.default_rng(4)
    B, K, V = 200, 5, 37
    z = rng.integers(-3, 4, size=(B, K + 1, V)).astype(np.float32)   # heavy ties
    g = np.argmax(z, axis=-1)                                        # first occurrence
    d = np.where(rng.random((B, K)) < 0.7, g[:, :K], rng.integers(0, V, size=(B, K))).astype(np.int32)
    out = oracle.verify(torch.tensor(z), None, d, 0.0, seed=0)
    for b in range(B):
        j = 0
        while j < K and d[b, j] == g[b, j]:
            j += 1
        assert out["accept_len"][b] == j
        assert list(out["tokens"][b, :j]) == list(d[b, :j])
        assert out["tokens"][b, j] == g[b, j]
        assert (out["tokens"][b, j + 1:] == -1).all()


def test_bf16_inputs_convert_exactly():
    z32 = torch.tensor([[[0.5, -1.25, 3.0, -math.inf]]], dtype=torch.float32).expand(1, 2, 4).contiguous()
    zb = z32.to(torch.bfloat16)
    d = torch.tensor([[2]], dtype=torch.int32)
    a = oracle.verify(z32, z32[:, :1].clone(), d, 0.8, seed=1, full=True)
    b = oracle.verify(zb, zb[:, :1].clone(), d, 0.8, seed=1, full=True)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])
    np.testing.assert_array_equal(a["row_lse"], b["row_lse"])


def test_data_errors():
    B, K, V = 6, 3, 16
    rng = np.random.default_rng(2)
    zt = torch.tensor(rng.normal(0, 1, size=(B, K + 1, V)), dtype=torch.float32)
    zd = zt[:, :K].clone()
    d = torch.tensor(rng.integers(0, V, size=(B, K)), dtype=torch.int32)
    zt[0, 0, 3] = math.nan
    zt[1, 0, :] = -math.inf
    d[2, 0] = V
    zd[3, 0, 5] = math.inf
    zt[4, K, 1] = math.nan            # bonus row, reached because p == q elsewhere
    zt[5, K - 1, 0] = math.nan        # never examined? p == q => all accepted => examined
    out = oracle.verify(zt, zd, d, 1.0, seed=3)
    assert list(out["accept_len"]) == [-2, -2, -3, -2, -2, -2]
    assert (out["tokens"] == -1).all()


def test_shortlist_equals_full_vocab_with_minus_inf():
    """A draft defined on a shortlist equals the full-vocabulary draft with
    -inf off the shortlist (the DynaSpec summary: verification keeps the full
    vocabulary)."""
    rng = np.random.default_rng(6)
    B, K, V, S = 40, 3, 64, 16
    zt = torch.tensor(rng.normal(0, 2, size=(B, K + 1, V)), dtype=torch.float32)
    sl = torch.tensor(np.stack([np.sort(rng.choice(V, S, replace=False)) for _ in range(B)]),
                      dtype=torch.int32)
    comp = torch.gather(zt[:, :K], 2, sl.long().unsqueeze(1).expand(B, K, S)) + 0.3
    full = torch.full((B, K, V), -math.inf)
    full.scatter_(2, sl.long().unsqueeze(1).expand(B, K, S), comp)
    d = torch.gather(sl, 1, torch.tensor(rng.integers(0, S, size=(B, K))))
    a = oracle.verify(zt, comp, d, 1.0, seed=8, shortlist=sl, full=True)
    b = oracle.verify(zt, full, d, 1.0, seed=8, full=True)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])
    np.testing.assert_array_equal(a["accept_len"], b["accept_len"])
    np.testing.assert_allclose(a["q_draft"], b["q_draft"], atol=1e-15)
    np.testing.assert_allclose(a["p_draft"], b["p_draft"], atol=1e-15)
    bad = sl.clone()
    bad[0, 3] = bad[0, 2]
    c = oracle.verify(zt, comp, d, 1.0, seed=8, shortlist=bad)
    assert c["accept_len"][0] == -4


def test_draft_probability_errors_only_where_read():
    """Given draft probabilities are used at p_i(d_i) for the accept test and
    as a whole row only at a rejection: a bad entry elsewhere in an accepted
    position's row is never read."""
    B, K, V = 3, 2, 8
    q = np.full(V, 1.0 / V)
    p = np.full(V, 1.0 / V)
    tgt, drf = _batch([q, q, q], [p, p], np.zeros((B, K), dtype=np.int32))
    drf = drf.clone()
    d = torch.zeros((B, K), dtype=torch.int32)
    drf[0, 0, 5] = -0.25     # p == q elsewhere: position 1 accepted, entry 5 never read
    drf[1, 0, 0] = math.nan  # the drafted token's own probability: read at position 1
    drf[2, 0, 0] = 0.25      # q/p = 0.5: some seeds reject, then the row is read
    drf[2, 0, 3] = math.inf
    out = oracle.verify(tgt, drf, d, 1.0, seed=2, draft_is_probs=True)
    assert out["accept_len"][0] == K
    assert out["accept_len"][1] == -2
    outs = [oracle.verify(tgt, drf, d, 1.0, seed=s, draft_is_probs=True)["accept_len"][2]
            for s in range(40)]
    assert -2 in outs and all(x in (-2, 1, 2) for x in outs)
