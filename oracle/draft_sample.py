"""Float64 oracle of the fused draft-token sampler.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``: only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may use it).

What it computes is the drafting step that precedes verification:
  - nextadmin.net lesson "Speculative Decoding", § Core algorithm, step 2: the
    draft model proposes d_1 .. d_N together with its probabilities p_1 .. p_N;
  - the same lesson, § Build it (``spec_step``): each drafted token is drawn
    from the draft distribution, and the probability of the drawn token,
    p_dist[d], is kept for the acceptance test;
  - aiengineeringfromscratch.com lesson 25, § Build it: the draft distribution
    is the softmax of the draft logits divided by the temperature.

Readings (the pages leave these open):
  - "sample" is the same inverse-CDF rule the verification oracle uses: the
    smallest x whose running sum of p in ascending token order exceeds v * R,
    R = sum(p) (so rounding in the normalisation cannot move the boundary);
  - v is word 0 of Philox4x32-10 with counter (position i, sequence b, tag 1
    (draft generation), 0) and key (seed low word, seed high word), mapped by
    ((w >> 8) + 0.5) * 2^-24;
  - each position is drawn from its own row of draft logits (the rows are the
    drafter's outputs, already conditioned on the earlier drafts);
  - T == 0 drafts greedily: the first index of the largest logit, with
    p_i(d_i) = 1 (the greedy drafter's distribution is one-hot);
  - a row with a NaN or +inf logit, or with every logit -inf, is an error:
    token -1, probability NaN.

Pinned in ``tests/test_oracle_draft_sample.py`` (closed form for uniform
logits, numpy.searchsorted on the normalised CDF, a chi-square test against the
softmax, temperature scaling, one-hot rows, greedy against numpy.argmax).
"""
from __future__ import annotations

import numpy as np

from . import BF16, F32, _raw, argmax_first, inverse_cdf, philox4x32_10, softmax, uniform24

TAG_DRAFT_GEN = 1
ERR_NONFINITE = 2


def row_f64(a: np.ndarray, dt: int) -> np.ndarray:
    """A row in the oracle's element codes as float64 (exact for both dtypes)."""
    if dt == BF16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dt == F32:
        return a.astype(np.float64)
    raise TypeError("unknown element code")


def draft_uniform(seed: int, seq: int, pos: int) -> float:
    key = [int(seed) & 0xffffffff, (int(seed) >> 32) & 0xffffffff]
    w = philox4x32_10([pos, seq, TAG_DRAFT_GEN, 0], key)
    return uniform24(int(w[0]))


def sample_row(z: np.ndarray, T: float, v: float):
    """One draw from softmax(z / T) with uniform v.
    Returns (token, probability of the token, margin, status)."""
    if T == 0.0:
        x = argmax_first(z)
        if x < 0:
            return -1, float("nan"), 0.0, ERR_NONFINITE
        return x, 1.0, float("inf"), 0
    try:
        p, _ = softmax(z, T)
    except ValueError:
        return -1, float("nan"), 0.0, ERR_NONFINITE
    x, margin = inverse_cdf(p, float(p.sum()), v)
    return x, float(p[x] / p.sum()), margin, 0


def draft_sample(draft, T: float, seed: int, seq_ids=None) -> dict:
    """draft: [B][K][V] float32 or bfloat16 logits (torch tensor or numpy:
    float32, or uint16 bfloat16 bits).  ``seq_ids`` [B] gives the sequence
    index that keys each row's uniforms (default: the row number).
    Returns numpy arrays tokens [B][K] int32, prob [B][K] float64,
    margin [B][K] (distance of v to the nearer edge of the drawn token's CDF
    interval) and status [B][K]."""
    a, dt = _raw(draft)
    B, K, V = a.shape
    sid = np.arange(B) if seq_ids is None else np.asarray(seq_ids)
    tokens = np.full((B, K), -1, dtype=np.int32)
    prob = np.full((B, K), np.nan)
    margin = np.zeros((B, K))
    status = np.zeros((B, K), dtype=np.int32)
    for b in range(B):
        for i in range(K):
            v = draft_uniform(seed, int(sid[b]), i)
            x, pr, m, st = sample_row(row_f64(a[b, i], dt), T, v)
            tokens[b, i], prob[b, i], margin[b, i], status[b, i] = x, pr, m, st
    return dict(tokens=tokens, prob=prob, margin=margin, status=status)
