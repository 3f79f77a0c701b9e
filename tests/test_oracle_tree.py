"""Pins for the greedy tree-verification oracle and the tree mask: the
page's tree figure (golden topology), the chain tree as the ordinary greedy
rule (already pinned against numpy.argmax), brute-force enumeration of root
paths, and the mask against the ancestor relation and the causal mask."""
from __future__ import annotations

import itertools
import json
import os

import numpy as np
import torch

import oracle
from oracle import tree as ot

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_figure.json")


def _logits_with_argmax(N, V, argmax, gen):
    z = torch.randn((N, V), generator=gen)
    for n, x in argmax.items():
        z[n, x] = 10.0
    return z


def test_figure_tree_longest_accepted_branch():
    g = json.load(open(GOLDEN))
    parent = np.array(g["parent"])
    N, V = len(parent), 50
    names = g["names"]
    tok = {"a": 5, "b": 6, "c": 7, "d": 8, "e": 9, "f": 10}
    tokens = np.array([0] + [tok[n] for n in names[1:]])
    gen = torch.Generator().manual_seed(0)
    # the target picks a after the root and d after a; its pick after d is the bonus
    z = _logits_with_argmax(N, V, {0: tok["a"], 1: tok["d"], 4: 33, 2: tok["e"]}, gen)
    out = ot.tree_verify_greedy(z[None], tokens[None], parent[None])
    assert out["accept_len"][0] == 2
    assert out["tokens"][0, :3].tolist() == [tok["a"], tok["d"], 33]
    assert [names[n] for n in out["nodes"][0, :2]] == g["ancestors_of_d"][1:]
    m = ot.tree_mask(parent)
    d = names.index("d")
    assert [names[j] for j in np.nonzero(m[d])[0]] == g["ancestors_of_d"]
    assert m.sum(1).tolist() == [x + 1 for x in g["depth"]]


def test_chain_tree_is_the_greedy_rule():
    gen = torch.Generator().manual_seed(1)
    B, K, V = 6, 5, 40
    z = torch.randint(0, 6, (B, K + 1, V), generator=gen).float()      # many ties
    best = z.argmax(-1)
    drafts = torch.where(torch.rand((B, K), generator=gen) < 0.7, best[:, :K],
                         torch.randint(0, V, (B, K), generator=gen)).to(torch.int32)
    ref = oracle.verify(z, None, drafts, 0.0, 0)
    tokens = np.concatenate([np.zeros((B, 1), np.int32), drafts.numpy()], 1)
    parent = np.tile(np.arange(-1, K), (B, 1))
    out = ot.tree_verify_greedy(z, tokens, parent)
    assert np.array_equal(out["accept_len"], ref["accept_len"])
    assert np.array_equal(out["tokens"][:, :K + 1], ref["tokens"])
    assert np.array_equal(ot.tree_mask(parent[0]), np.tril(np.ones((K + 1, K + 1), np.uint8)))


def _brute(z, tokens, parent):
    """Every root path; the deepest one whose edges all match the argmax."""
    N = len(parent)
    g = z.argmax(-1).tolist()
    best = (0, 0)
    for n in range(1, N):
        path, m = [], n
        while m > 0:
            path.append(m)
            m = parent[m]
        if all(tokens[c] == g[parent[c]] for c in path):
            best = max(best, (len(path), -n))
    n = -best[1]
    return best[0], g[n]


def test_random_trees_against_brute_force():
    gen = torch.Generator().manual_seed(2)
    rng = np.random.default_rng(2)
    for trial in range(40):
        N, V = int(rng.integers(2, 14)), int(rng.integers(3, 7))
        parent = np.array([-1] + [int(rng.integers(0, n)) for n in range(1, N)])
        z = torch.randn((N, V), generator=gen)
        tokens = rng.integers(0, V, N)
        depth, bonus = _brute(z.numpy(), tokens, parent)
        out = ot.tree_verify_greedy(z[None], tokens[None], parent[None])
        assert out["accept_len"][0] == depth
        assert out["tokens"][0, depth] == bonus
        # the mask: ancestors by brute force
        m = ot.tree_mask(parent)
        for i, j in itertools.product(range(N), range(N)):
            anc, k = False, i
            while k >= 0:
                anc |= k == j
                k = parent[k] if k > 0 else -1
            assert m[i, j] == anc


def test_errors_only_where_examined():
    gen = torch.Generator().manual_seed(3)
    parent = np.array([-1, 0, 0, 1, 2])
    z = _logits_with_argmax(5, 20, {0: 4, 1: 9}, gen)
    tokens = np.array([0, 4, 7, 3, 99])       # node 4's token is out of range, but node 2 is rejected
    z[2, 0] = float("nan")                   # node 2's row is never examined
    out = ot.tree_verify_greedy(z[None], tokens[None], parent[None])
    assert out["accept_len"][0] == 1 and out["tokens"][0, :2].tolist() == [4, 9]
    z[1, 3] = float("inf")                   # node 1 is accepted: its row is examined
    out = ot.tree_verify_greedy(z[None], tokens[None], parent[None])
    assert out["accept_len"][0] == -ot.ERR_NONFINITE
    bad = ot.tree_verify_greedy(z[None], tokens[None], np.array([[-1, 0, 3, 1, 2]]))
    assert bad["accept_len"][0] == -ot.ERR_TREE
