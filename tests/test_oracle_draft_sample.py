"""Pins for the draft-sampler oracle (``oracle.draft_sample``).

Each test checks the oracle against something other than itself: a closed
form, a library routine on the normalised CDF, the softmax it must sample
from (chi-square), temperature scaling, or numpy.argmax.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch
from scipy import stats

from oracle import draft_sample as ds


def _np_softmax(z, T):
    z = np.asarray(z, dtype=np.float64) / T
    m = np.max(z[np.isfinite(z)])
    e = np.where(np.isfinite(z), np.exp(z - m), 0.0)
    return e / e.sum()


def test_uniform_logits_closed_form():
    # equal logits: p = 1/V, so the inverse CDF gives floor(v * V)
    V, B, K = 1000, 64, 3
    z = torch.full((B, K, V), 0.75, dtype=torch.float32)
    out = ds.draft_sample(z, 1.3, seed=11)
    for b in range(B):
        for i in range(K):
            v = ds.draft_uniform(11, b, i)
            if abs(v * V - round(v * V)) < 1e-9:
                continue   # on a boundary: rounding decides
            assert out["tokens"][b, i] == math.floor(v * V)
            assert out["prob"][b, i] == pytest.approx(1.0 / V, rel=1e-12)


def test_matches_searchsorted_on_normalised_cdf():
    g = torch.Generator().manual_seed(3)
    B, K, V = 16, 4, 777
    z = 2.0 * torch.randn((B, K, V), generator=g)
    T = 0.8
    out = ds.draft_sample(z, T, seed=5)
    for b in range(B):
        for i in range(K):
            p = _np_softmax(z[b, i].double().numpy(), T)
            v = ds.draft_uniform(5, b, i)
            x = int(np.searchsorted(np.cumsum(p), v * p.sum(), side="right"))
            if out["margin"][b, i] > 1e-12:
                assert out["tokens"][b, i] == x
            assert out["prob"][b, i] == pytest.approx(p[out["tokens"][b, i]], rel=1e-9)


def test_chi_square_against_softmax():
    # one row of 8 logits repeated over 40000 sequences: the histogram of the
    # drawn tokens follows softmax(z / T)
    z8 = torch.tensor([1.0, -0.5, 0.3, 2.0, -1.0, 0.0, 0.7, -2.0])
    T = 0.9
    B = 40000
    out = ds.draft_sample(z8.reshape(1, 1, 8).expand(B, 1, 8).contiguous(), T, seed=2024)
    counts = np.bincount(out["tokens"][:, 0], minlength=8)
    exp = _np_softmax(z8.numpy(), T) * B
    assert stats.chisquare(counts, exp).pvalue > 0.001


def test_temperature_divides_the_logits():
    # drawing at temperature T from z is drawing at temperature 1 from z / T
    g = torch.Generator().manual_seed(9)
    z = torch.randn((8, 2, 300), generator=g, dtype=torch.float64).float()
    T = 0.5
    a = ds.draft_sample(z, T, seed=77)
    b = ds.draft_sample((z.double() / T).float(), 1.0, seed=77)
    ok = (a["margin"] > 1e-9) & (b["margin"] > 1e-9)
    assert ok.sum() > 10
    assert np.array_equal(a["tokens"][ok], b["tokens"][ok])


def test_one_hot_row_is_deterministic():
    V = 50
    z = torch.full((4, 2, V), -math.inf)
    z[:, :, 17] = 3.0
    out = ds.draft_sample(z, 1.0, seed=1)
    assert (out["tokens"] == 17).all()
    assert np.allclose(out["prob"], 1.0)


def test_greedy_is_numpy_argmax_first():
    g = torch.Generator().manual_seed(4)
    z = torch.randint(0, 5, (6, 3, 40), generator=g).float()   # many ties
    out = ds.draft_sample(z, 0.0, seed=0)
    assert np.array_equal(out["tokens"], np.argmax(z.numpy(), axis=-1))
    assert (out["prob"] == 1.0).all()


def test_bf16_rows_convert_exactly():
    g = torch.Generator().manual_seed(8)
    z = torch.randn((3, 2, 64), generator=g).to(torch.bfloat16)
    a = ds.draft_sample(z, 1.0, seed=3)
    b = ds.draft_sample(z.float(), 1.0, seed=3)
    assert np.array_equal(a["tokens"], b["tokens"])
    assert np.array_equal(a["prob"], b["prob"])


def test_errors():
    z = torch.zeros((1, 3, 10))
    z[0, 0, 4] = math.nan
    z[0, 1, :] = -math.inf
    z[0, 2, 2] = math.inf
    out = ds.draft_sample(z, 1.0, seed=0)
    assert (out["tokens"] == -1).all()
    assert (out["status"] == ds.ERR_NONFINITE).all()
    assert np.isnan(out["prob"]).all()
