"""Greedy tree verification and the tree mask (CUDA, through the C ABI)
against the oracle: bit-exact tokens, nodes, lengths and masks."""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

import speculative_decoding_verification_sampling_gb300 as sv
from oracle import tree as ot
from speculative_decoding_verification_sampling_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_figure.json")


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(DEV)
    sv.load()


def _check(target, tokens, parent, status_expected=None):
    st = torch.full((1,), -3, dtype=torch.int32, device=DEV)
    t, n, l = sv.spec_verify_tree_greedy(target.to(DEV).contiguous(), tokens.to(DEV).to(torch.int32).contiguous(),
                                         parent.to(DEV).to(torch.int32).contiguous(), device_status=st)
    ref = ot.tree_verify_greedy(target, tokens.numpy(), parent.numpy())
    assert np.array_equal(l.cpu().numpy(), ref["accept_len"])
    ok = ref["accept_len"] >= 0
    assert np.array_equal(t.cpu().numpy()[ok], ref["tokens"][ok])
    assert np.array_equal(n.cpu().numpy()[ok], ref["nodes"][ok])
    if status_expected is not None:
        assert int(st.item()) == status_expected
    return ref


@pytest.mark.parametrize("B,V,branching,dtype", [
    (8, 128256, (4, 2, 2, 1, 1), torch.bfloat16),
    (3, 32000, (2, 2, 2), torch.float32),
    (5, 1001, (3, 3, 1), torch.bfloat16),      # rows not 16-byte aligned
    (2, 7, (3, 2), torch.float32),            # fewer tokens than one vector
])
def test_tree_matches_oracle(B, V, branching, dtype):
    cfg = synth.tree_greedy(B=B, V=V, branching=branching, dtype=dtype, seed=B + V % 13)
    ref = _check(cfg["target"], cfg["tree_tokens"], cfg["parent"], 0)
    assert (ref["accept_len"] >= 0).all()


def test_figure_tree():
    g = json.load(open(GOLDEN))
    parent = torch.tensor(g["parent"], dtype=torch.int32)[None]
    z = torch.randn((1, 7, 64))
    z[0, 0, 5] = 9.0
    z[0, 1, 8] = 9.0
    tokens = torch.tensor([[0, 5, 6, 7, 8, 9, 10]], dtype=torch.int32)
    ref = _check(z, tokens, parent, 0)
    assert ref["accept_len"][0] == 2
    m = sv.spec_tree_mask(parent.to(DEV)).cpu().numpy()[0]
    assert np.array_equal(m, ot.tree_mask(g["parent"]))


def test_heavy_ties_and_chain():
    g = torch.Generator().manual_seed(5)
    B, K, V = 16, 6, 300
    z = torch.randint(0, 3, (B, K + 1, V), generator=g).float()
    best = z.argmax(-1)
    tokens = torch.cat([torch.zeros(B, 1, dtype=torch.long),
                        torch.where(torch.rand(B, K, generator=g) < 0.8, best[:, :K],
                                    torch.randint(0, V, (B, K), generator=g))], 1)
    parent = torch.arange(-1, K).expand(B, K + 1)
    _check(z, tokens, parent, 0)


def test_errors():
    g = torch.Generator().manual_seed(6)
    B, V = 4, 100
    parent = torch.tensor([-1, 0, 0, 1, 2], dtype=torch.int32).expand(B, 5).clone()
    z = torch.randn((B, 5, V), generator=g)
    z[:, 0, 4] = 20.0
    tokens = torch.tensor([0, 4, 7, 3, 99], dtype=torch.int32).expand(B, 5).clone()
    z[1, 1, 3] = math.inf           # b=1: accepted node 1's row is bad
    z[2, 2, 0] = math.nan           # b=2: node 2 is rejected, its row is never examined
    parent[3, 2] = 5                # b=3: malformed tree
    ref = _check(z, tokens, parent)
    assert ref["accept_len"].tolist()[1] == -2 and ref["accept_len"].tolist()[3] == -1
    assert ref["accept_len"][0] >= 0 and ref["accept_len"][2] >= 0


@pytest.mark.parametrize("branching", [(4, 2, 2, 1, 1), (8,), (1, 1, 1, 1, 1, 1, 1), (3, 3, 3, 3)])
def test_mask_matches_oracle(branching):
    parent = torch.tensor(synth.tree_topology(branching), dtype=torch.int32)
    B = 3
    par = parent.expand(B, -1).contiguous()
    m = sv.spec_tree_mask(par.to(DEV)).cpu().numpy()
    want = ot.tree_mask(parent.numpy())
    for b in range(B):
        assert np.array_equal(m[b], want)


def test_mask_reports_malformed_parents():
    par = torch.tensor([[-1, 0, 3, 1]], dtype=torch.int32, device=DEV)
    st = torch.full((1,), -4, dtype=torch.int32, device=DEV)
    sv.spec_tree_mask(par, device_status=st)
    assert int(st.item()) == 1


def test_token_error_under_accepted_parent():
    # node 1 (the argmax of row 0) is accepted; its child, node 3, carries a
    # token outside [0, V): SPEC_ERR_TOKEN_RANGE.  A bad token under a rejected
    # node (node 4, under node 2) is never examined.
    g = torch.Generator().manual_seed(7)
    B, V = 3, 100
    parent = torch.tensor([-1, 0, 0, 1, 2], dtype=torch.int32).expand(B, 5).clone()
    z = torch.randn((B, 5, V), generator=g)
    z[:, 0, 4] = 20.0
    tokens = torch.tensor([0, 4, 7, 50, 60], dtype=torch.int32).expand(B, 5).clone()
    tokens[0, 3] = V + 5
    tokens[1, 4] = -7
    tokens[2, 3] = -1
    ref = _check(z, tokens, parent)
    assert ref["accept_len"].tolist() == [-3, ref["accept_len"][1], -3]
    assert ref["accept_len"][1] >= 0
