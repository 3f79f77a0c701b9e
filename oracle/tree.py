"""Oracle of greedy tree verification and of the tree attention mask.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``).

Source: aiengineeringfromscratch.com Phase 10 lesson 25 "Speculative
Decoding", § Tree attention verification (a draft tree is verified by one
target forward pass under a mask that lets each token attend only to its
ancestors; the output is the longest accepted prefix along any path) and
§ Greedy case (a draft token is accepted when it equals the target's argmax).
The stochastic multi-branch rule is not on the pages, so only the greedy rule
is defined here.

Tree layout (per sequence): N nodes in an order where every parent comes
before its children; node 0 is the root (the last token already accepted,
parent -1); node n >= 1 holds a drafted token tokens[n] and its parent
parent[n] < n.  Row n of the target logits is the target's prediction after
node n's token (computed under the tree mask).

Readings:
  - a child c of an accepted node n is accepted iff tokens[c] == argmax of
    row n (first index of the maximum of the raw logits); the root is
    accepted;
  - the longest accepted path ends at the deepest accepted node, the lowest
    node index among equally deep ones; the emitted tokens are the drafted
    tokens along that path followed by the argmax of its last node's row
    (the bonus of the greedy rule);
  - only the rows of accepted nodes are examined: a NaN or +inf (or an all
    -inf row) there is an error (code 2), as is a token outside [0, V) at a
    child of an accepted node (code 3); a malformed parent array (parent[0]
    != -1, or parent[n] not in [0, n)) is an error (code 1);
  - mask[i][j] = 1 iff node j is node i or one of its ancestors.
"""
from __future__ import annotations

import numpy as np

from . import argmax_first
from .draft_sample import row_f64
from . import _raw

ERR_TREE, ERR_NONFINITE, ERR_TOKEN = 1, 2, 3


def tree_ok(parent) -> bool:
    parent = np.asarray(parent)
    return parent.shape[0] >= 1 and parent[0] == -1 and all(0 <= parent[n] < n for n in range(1, parent.shape[0]))


def tree_mask(parent) -> np.ndarray:
    """[N][N] uint8: mask[i][j] = 1 iff j is i or an ancestor of i."""
    parent = np.asarray(parent)
    N = parent.shape[0]
    m = np.zeros((N, N), dtype=np.uint8)
    for i in range(N):
        j = i
        while j >= 0:
            m[i, j] = 1
            j = parent[j] if j > 0 else -1
    return m


def tree_verify_greedy(target, tokens, parent) -> dict:
    """target [B][N][V] float32 or bfloat16 logits; tokens, parent [B][N].
    Returns tokens [B][N] (path tokens then the bonus, -1 after), nodes [B][N]
    (the path's node indices, root excluded, -1 after) and accept_len [B]
    (-code on error)."""
    a, dt = _raw(target)
    B, N, V = a.shape
    tokens = np.asarray(tokens).reshape(B, N)
    parent = np.asarray(parent).reshape(B, N)
    out_t = np.full((B, N), -1, dtype=np.int32)
    out_n = np.full((B, N), -1, dtype=np.int32)
    out_l = np.zeros(B, dtype=np.int32)
    for b in range(B):
        if not tree_ok(parent[b]):
            out_l[b] = -ERR_TREE
            continue
        g = {}
        acc = np.zeros(N, dtype=bool)
        acc[0] = True
        depth = np.zeros(N, dtype=np.int64)
        err = 0
        for n in range(N):
            if n > 0:
                p = parent[b, n]
                depth[n] = depth[p] + 1
                if not acc[p]:
                    continue
                if not (0 <= tokens[b, n] < V):
                    err = ERR_TOKEN
                    break
                acc[n] = tokens[b, n] == g[p]
                if not acc[n]:
                    continue
            x = argmax_first(row_f64(a[b, n], dt))
            if x < 0:
                err = ERR_NONFINITE
                break
            g[n] = x
        if err:
            out_l[b] = -err
            continue
        cand = [n for n in range(N) if acc[n]]
        best = min(cand, key=lambda n: (-depth[n], n))
        path = []
        n = best
        while n > 0:
            path.append(n)
            n = parent[b, n]
        path.reverse()
        for k, n in enumerate(path):
            out_t[b, k] = tokens[b, n]
            out_n[b, k] = n
        out_t[b, len(path)] = g[best]
        out_l[b] = len(path)
    return dict(tokens=out_t, nodes=out_n, accept_len=out_l)
