"""Exact output distribution of one verification round, by enumeration.

Used only to pin the float64 oracle on tiny vocabularies (V <= 4, K <= 2).
It is an independent statement of the outcome probabilities, in rational
arithmetic: for fixed draft tokens d_1..d_K, the round emits
  d_1..d_{j-1}, x   with probability  prod_{i<j} a_i * (1 - a_j) * r_j(x) / R_j
  d_1..d_K, x       with probability  prod_{i<=K} a_i * q_{K+1}(x)
where a_i = min(1, q_i(d_i) / p_i(d_i)) (1 when p_i(d_i) = 0) and
r_j = (q_j - p_j)_+ with total R_j (nextadmin.net lesson "Speculative
Decoding", core algorithm steps 4-6; aiengineeringfromscratch.com lesson 25,
"the exact rule").  Enumerating d_i ~ p_i gives the marginal distribution,
whose first token must equal q_1 exactly (the distribution-preservation
theorem the pages state) -- that identity pins this module itself.
"""
from __future__ import annotations

from collections import defaultdict
from fractions import Fraction
from itertools import product


def accept_probability(q_d: Fraction, p_d: Fraction) -> Fraction:
    if p_d == 0:
        return Fraction(1)
    return min(Fraction(1), q_d / p_d)


def round_given_drafts(q, p, drafts) -> dict:
    """q: K+1 distributions, p: K distributions (lists of Fraction); drafts: K tokens.
    Returns {emitted token tuple: probability}."""
    K = len(p)
    out = defaultdict(Fraction)
    reach = Fraction(1)
    for i, d in enumerate(drafts):
        a = accept_probability(q[i][d], p[i][d])
        stop = reach * (1 - a)
        if stop:
            r = [max(Fraction(0), qx - px) for qx, px in zip(q[i], p[i])]
            R = sum(r)
            if R == 0:
                r, R = list(q[i]), sum(q[i])
            for x, rx in enumerate(r):
                if rx:
                    out[tuple(drafts[:i]) + (x,)] += stop * rx / R
        reach *= a
        if reach == 0:
            return dict(out)
    for x, qx in enumerate(q[K]):
        if qx:
            out[tuple(drafts) + (x,)] += reach * qx
    return dict(out)


def round_distribution(q, p) -> dict:
    """Marginal over independent draft tokens d_i ~ p_i."""
    K, V = len(p), len(q[0])
    total = defaultdict(Fraction)
    for drafts in product(range(V), repeat=K):
        w = Fraction(1)
        for i, d in enumerate(drafts):
            w *= p[i][d]
        if w == 0:
            continue
        for seq, pr in round_given_drafts(q, p, drafts).items():
            total[seq] += w * pr
    return dict(total)


def first_token_marginal(dist: dict, V: int) -> list:
    m = [Fraction(0)] * V
    for seq, pr in dist.items():
        m[seq[0]] += pr
    return m


def next_token_conditional(dist: dict, prefix: tuple, V: int):
    """Distribution of the token after `prefix` among rounds that emit more than len(prefix) tokens
    starting with `prefix`; None if no such round has positive probability."""
    n = len(prefix)
    m = [Fraction(0)] * V
    for seq, pr in dist.items():
        if len(seq) > n and seq[:n] == prefix:
            m[seq[n]] += pr
    tot = sum(m)
    if tot == 0:
        return None
    return [x / tot for x in m]
