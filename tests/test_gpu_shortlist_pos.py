"""Per-position shortlists (CUDA, through the C ABI) against the oracle:
sampled tokens identical except near-threshold uniforms (counted), residual
mass and per-position outputs within 1e-5; per-position, per-sequence and
shared lists; errors where the rule reaches them."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_sampling_gb300 as sv
from parity import assert_parity
from speculative_decoding_verification_sampling_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(DEV)
    sv.load()


def _run(cfg, seed, full=False, lists=None):
    lists = cfg["shortlist"] if lists is None else lists
    aux = sv.Aux.alloc(cfg["B"], cfg["K"], DEV, full=full)
    t, l = sv.spec_verify_shortlist_pos(cfg["target"].to(DEV), cfg["draft"].to(DEV), lists.to(DEV),
                                        cfg["draft_tokens"].to(DEV), cfg["T"], seed,
                                        shortlist_len=cfg.get("shortlist_len"), aux=aux)
    ref = oracle.verify(cfg["target"], cfg["draft"], cfg["draft_tokens"], cfg["T"], seed, shortlist=lists,
                        shortlist_len=cfg.get("shortlist_len"), full=full)
    return t.cpu().numpy(), l.cpu().numpy(), aux, ref


@pytest.mark.parametrize("B,K,V,n_clusters,budget,dtype", [
    (16, 6, 262144, 64, None, torch.bfloat16),
    (12, 4, 32000, 50, [5, 5, 2, 1], torch.float32),
    (20, 5, 4096, 32, [6, 3, 2, 1, 1], torch.bfloat16),
    (40, 3, 50000, 100, [4, 2, 1], torch.bfloat16),       # ragged last segment (50000 = 195 * 256 + 80)
])
def test_per_position_lists(B, K, V, n_clusters, budget, dtype):
    cfg = synth.shortlist_per_position(B=B, K=K, V=V, n_clusters=n_clusters, budget=budget, dtype=dtype,
                                       seed=B + K)
    t, l, aux, ref = _run(cfg, 31 + B, full=True)
    assert_parity(t, l, ref, "per-position shortlists")
    ok = ref["accept_len"] >= 0
    for name in ("q_draft", "p_draft", "row_lse"):
        g = getattr(aux, name).cpu().numpy()
        assert np.allclose(g[ok], ref[name][ok], atol=1e-5, rtol=0, equal_nan=True), name
    same = (l == ref["accept_len"]) & (t == ref["tokens"]).all(1)
    rm = aux.residual_mass.cpu().numpy()
    assert np.allclose(rm[same], ref["residual_mass"][same], atol=1e-5, rtol=0)


def test_sequence_and_shared_lists():
    cfg = synth.shortlist_per_position(B=24, K=4, V=20000, n_clusters=40, budget=[4, 4, 4, 4], seed=3)
    per_seq = cfg["shortlist"][:, 0].contiguous()                 # [B][S]: position 0's list everywhere
    d = cfg["draft"].clone()
    for i in range(cfg["K"]):
        d[:, i] = torch.gather(cfg["target"][:, i].float(), 1, per_seq.long()).to(d.dtype)
    c2 = dict(cfg, draft=d, shortlist_len=None)
    t, l, _, ref = _run(c2, 5, lists=per_seq)
    assert_parity(t, l, ref, "per-sequence lists")
    shared = per_seq[0].contiguous()                              # [S]: one list for all
    d2 = torch.stack([torch.stack([cfg["target"][b, i].float()[shared.long()] for i in range(cfg["K"])])
                      for b in range(cfg["B"])]).to(d.dtype)
    c3 = dict(cfg, draft=d2, shortlist_len=None)
    t, l, _, ref = _run(c3, 6, lists=shared)
    assert_parity(t, l, ref, "shared list")


def _gauss_case(seed, B=64, K=4, V=600, S=128):
    """Target ~ N(0, 1.5^2); random per-position lists of S, S, S/2, S/4 tokens;
    draft = target + N(0, 0.5^2) on each list; drafted tokens mostly on the list."""
    g = torch.Generator().manual_seed(seed)
    target = 1.5 * torch.randn((B, K + 1, V), generator=g)
    lens = [S, S, S // 2, S // 4][:K]
    lists = torch.zeros((B, K, S), dtype=torch.int32)
    draft = torch.zeros((B, K, S))
    tokens = torch.zeros((B, K), dtype=torch.int32)
    for b in range(B):
        for i in range(K):
            lst = torch.sort(torch.randperm(V, generator=g)[:lens[i]]).values
            lists[b, i, :lens[i]] = lst.to(torch.int32)
            draft[b, i, :lens[i]] = target[b, i, lst] + 0.5 * torch.randn(lens[i], generator=g)
            tokens[b, i] = int(lst[torch.argmax(draft[b, i, :lens[i]])])
    return dict(target=target, draft=draft, draft_tokens=tokens, T=1.0, shortlist=lists, shortlist_len=lens,
                B=B, K=K, V=V, S=S)


def test_bad_list_where_reached():
    cfg = _gauss_case(9)
    bad = cfg["shortlist"].clone()
    bad[:, 2, 1] = bad[:, 2, 0]
    t, l, _, ref = _run(cfg, 13, lists=bad)
    assert (ref["accept_len"] == -4).any() and (ref["accept_len"] >= 0).any()
    assert np.array_equal(l[ref["accept_len"] == -4], ref["accept_len"][ref["accept_len"] == -4])
    assert_parity(t, l, ref, "bad list")


def test_legacy_shortlist_call_on_row_kernels():
    """spec_verify_shortlist (one list per sequence) at a size the row kernels serve."""
    cfg = synth.shortlist(B=40, K=6, V=65536, n_clusters=64, per_seq=8, seed=12)
    t, l = sv.spec_verify_shortlist(cfg["target"].to(DEV), cfg["draft"].to(DEV), cfg["shortlist"].to(DEV),
                                    cfg["draft_tokens"].to(DEV), 1.0, 21)
    ref = oracle.verify(cfg["target"], cfg["draft"], cfg["draft_tokens"], 1.0, 21, shortlist=cfg["shortlist"])
    assert_parity(t.cpu().numpy(), l.cpu().numpy(), ref, "per-sequence shortlist")
