"""Seeded synthetic inputs for the verification step.

Input generation only: this module holds none of the verification arithmetic
(no softmax, no acceptance rule, no residual, no inverse CDF), so that the CUDA
path and the float64 oracle can both be fed from it without sharing any of the
method.  Draft tokens are drawn with the Gumbel-max trick (argmax of the
scaled logits plus Gumbel noise), which samples exactly from softmax(z / T)
without computing it.

Workloads (all logits are drawn from a seeded ``torch.Generator`` on the
requested device, then cast to the stated dtype):

* ``small_stochastic``  B=1, K=4, V=32000, float32, T=1: target ~ N(0, 2^2),
  draft = target + N(0, 0.5^2), draft tokens sampled from the draft softmax.
* ``greedy``            B=64, K=5, V=128256, bfloat16, T=0: target ~ N(0, 3^2);
  each draft token is the target argmax with probability 0.8, else uniform.
* ``zipf``              B=32, K=7, V=152064, bfloat16, T=0.7: Zipf-shaped
  logits -1.1 ln(rank) + N(0, 0.3^2), rank order permuted per row; draft =
  target + N(0, sigma^2), sigma in {0.25, 0.5, 1.0}.
* ``shortlist``         B=64, K=6, V=262144, bfloat16, T=1: vocabulary split at
  random into 64 clusters of 4096; each sequence draws 8 clusters (a sorted
  32768-token shortlist); target is full-vocabulary Zipf, the draft is
  target + N(0, 0.5^2) on the shortlist only (compact [B][K][S] layout).
* ``throughput``        B in {1, 8, 64, 256, 512}, K in {4, 8}, V=128256,
  bfloat16, T=1: target ~ N(0, 2^2), draft = target + N(0, 0.5^2).

The vocabulary sizes follow the pages' list of model vocabularies (32k Llama-2,
128k Llama-3, 152k Qwen-2.5, 262k Gemma-3 in the DynaSpec summary) and the
shortlist size follows its FR-Spec 32k / DynaSpec 27.3k comparison.  No public
benchmark data is used: these synthetic inputs stand in for the datasets and
trained models the pages measured with.
"""
from __future__ import annotations

import math

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gumbel_max_tokens(logits: torch.Tensor, T: float, gen: torch.Generator,
                      row_chunk: int = 256) -> torch.Tensor:
    """One token per row of ``logits`` (any leading shape), drawn from
    softmax(logits / T) by the Gumbel-max trick.  Returns int32."""
    lead = logits.shape[:-1]
    z = logits.reshape(-1, logits.shape[-1])
    out = torch.empty(z.shape[0], dtype=torch.int64, device=z.device)
    for r0 in range(0, z.shape[0], row_chunk):
        blk = z[r0:r0 + row_chunk].float()
        u = torch.rand(blk.shape, generator=gen, device=z.device, dtype=torch.float32)
        u.clamp_(min=1e-30, max=1.0 - 2.0 ** -24)
        g = -torch.log(-torch.log(u))
        out[r0:r0 + row_chunk] = torch.argmax(blk / T + g, dim=-1)
    return out.reshape(lead).to(torch.int32)


def zipf_logits(rows: int, V: int, gen: torch.Generator, device, noise_std: float = 0.3,
                exponent: float = 1.1, row_chunk: int = 64) -> torch.Tensor:
    """Float32 [rows][V]: -exponent * ln(rank) + N(0, noise_std^2), with the
    rank order randomly permuted per row."""
    base = -exponent * torch.log(torch.arange(1, V + 1, device=device, dtype=torch.float32))
    out = torch.empty((rows, V), device=device, dtype=torch.float32)
    for r0 in range(0, rows, row_chunk):
        n = min(row_chunk, rows - r0)
        perm = torch.argsort(torch.rand((n, V), generator=gen, device=device), dim=1)
        blk = torch.empty((n, V), device=device, dtype=torch.float32)
        blk.scatter_(1, perm, base.expand(n, V))
        blk += noise_std * torch.randn((n, V), generator=gen, device=device)
        out[r0:r0 + n] = blk
    return out


def _normal(shape, std, gen, device):
    return std * torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def stochastic_gaussian(B: int, K: int, V: int, dtype=torch.bfloat16, T: float = 1.0,
                        target_std: float = 2.0, draft_noise: float = 0.5, seed: int = 5,
                        device="cpu") -> dict:
    """Target ~ N(0, target_std^2); draft = target + N(0, draft_noise^2);
    draft tokens from the draft softmax at temperature T."""
    g = _gen(seed, device)
    target = _normal((B, K + 1, V), target_std, g, device).to(dtype)
    draft = (target[:, :K].float() + _normal((B, K, V), draft_noise, g, device)).to(dtype)
    tokens = gumbel_max_tokens(draft, T, g)
    return dict(name=f"stochastic B={B} K={K} V={V} {str(dtype).replace('torch.', '')} T={T}",
                target=target, draft=draft, draft_tokens=tokens, T=T, shortlist=None,
                B=B, K=K, V=V)


def small_stochastic(seed: int = 1, device="cpu") -> dict:
    d = stochastic_gaussian(1, 4, 32000, torch.float32, 1.0, 2.0, 0.5, seed, device)
    d["name"] = "stochastic B=1 K=4 V=32000 f32 T=1"
    return d


def greedy(B: int = 64, K: int = 5, V: int = 128256, dtype=torch.bfloat16, seed: int = 2,
           device="cpu", match_prob: float = 0.8, target_std: float = 3.0) -> dict:
    g = _gen(seed, device)
    target = _normal((B, K + 1, V), target_std, g, device).to(dtype)
    best = torch.argmax(target[:, :K].float(), dim=-1)
    rand_tok = torch.randint(0, V, (B, K), generator=g, device=device)
    keep = torch.rand((B, K), generator=g, device=device) < match_prob
    tokens = torch.where(keep, best, rand_tok).to(torch.int32)
    return dict(name=f"greedy B={B} K={K} V={V} {str(dtype).replace('torch.', '')}",
                target=target, draft=None, draft_tokens=tokens, T=0.0, shortlist=None,
                B=B, K=K, V=V)


def zipf(sigma: float = 0.5, B: int = 32, K: int = 7, V: int = 152064, dtype=torch.bfloat16,
         T: float = 0.7, seed: int = 3, device="cpu") -> dict:
    g = _gen(seed, device)
    target = zipf_logits(B * (K + 1), V, g, device).reshape(B, K + 1, V).to(dtype)
    draft = (target[:, :K].float() + _normal((B, K, V), sigma, g, device)).to(dtype)
    tokens = gumbel_max_tokens(draft, T, g)
    return dict(name=f"zipf B={B} K={K} V={V} sigma={sigma} T={T}", target=target, draft=draft,
                draft_tokens=tokens, T=T, shortlist=None, B=B, K=K, V=V)


def random_shortlists(B: int, V: int, n_clusters: int, per_seq: int, gen, device) -> torch.Tensor:
    """[B][S] int32, each row the sorted union of `per_seq` clusters drawn
    uniformly from a random partition of the vocabulary into `n_clusters`."""
    assert V % n_clusters == 0
    size = V // n_clusters
    perm = torch.randperm(V, generator=gen, device=device)
    clusters = perm.reshape(n_clusters, size)
    rows = []
    for _ in range(B):
        pick = torch.randperm(n_clusters, generator=gen, device=device)[:per_seq]
        rows.append(torch.sort(clusters[pick].reshape(-1)).values)
    return torch.stack(rows).to(torch.int32)


def shortlist(B: int = 64, K: int = 6, V: int = 262144, n_clusters: int = 64, per_seq: int = 8,
              dtype=torch.bfloat16, T: float = 1.0, sigma: float = 0.5, seed: int = 4,
              device="cpu") -> dict:
    g = _gen(seed, device)
    target = zipf_logits(B * (K + 1), V, g, device).reshape(B, K + 1, V).to(dtype)
    sl = random_shortlists(B, V, n_clusters, per_seq, g, device)
    idx = sl.long().unsqueeze(1).expand(B, K, sl.shape[1])
    draft = (torch.gather(target[:, :K].float(), 2, idx)
             + _normal((B, K, sl.shape[1]), sigma, g, device)).to(dtype)
    pos = gumbel_max_tokens(draft, T, g).long()
    tokens = torch.gather(sl.long(), 1, pos).to(torch.int32)
    return dict(name=f"shortlist B={B} K={K} V={V} S={sl.shape[1]}", target=target, draft=draft,
                draft_tokens=tokens, T=T, shortlist=sl, B=B, K=K, V=V)


def throughput(B: int = 256, K: int = 4, seed: int = 5, device="cpu") -> dict:
    d = stochastic_gaussian(B, K, 128256, torch.bfloat16, 1.0, 2.0, 0.5, seed, device)
    d["name"] = f"stochastic B={B} K={K} V=128256 bf16 T=1"
    return d


def log_probs(prob: torch.Tensor) -> torch.Tensor:
    """Natural-log logits of a probability vector (-inf where the probability is 0)."""
    prob = prob.double()
    out = torch.full_like(prob, -math.inf)
    nz = prob > 0
    out[nz] = torch.log(prob[nz])
    return out


def controlled_alpha_pair(V: int, alpha: float, gen: torch.Generator):
    """A target q on the first half of the vocabulary and a draft
    p = alpha * q + (1 - alpha) * r with r on the other half, so that
    sum_x min(p(x), q(x)) == alpha.  Returns float64 (q, p)."""
    half = V // 2
    q = torch.zeros(V, dtype=torch.float64)
    r = torch.zeros(V, dtype=torch.float64)
    wq = torch.rand(half, generator=gen, dtype=torch.float64) + 0.1
    wr = torch.rand(V - half, generator=gen, dtype=torch.float64) + 0.1
    q[:half] = wq / wq.sum()
    r[half:] = wr / wr.sum()
    return q, alpha * q + (1.0 - alpha) * r


def tree_topology(branching=(4, 2, 2, 1, 1)) -> list[int]:
    """Parents of a draft tree in breadth-first order: the root, then
    `branching[0]` children, each with `branching[1]` children, and so on
    (EAGLE-style top-k branches per depth).  Node 0 is the root (parent -1)."""
    parent, level = [-1], [0]
    for k in branching:
        nxt = []
        for p in level:
            for _ in range(k):
                parent.append(p)
                nxt.append(len(parent) - 1)
        level = nxt
    return parent


def tree_greedy(B: int = 32, V: int = 128256, branching=(4, 2, 2, 1, 1), dtype=torch.bfloat16, seed: int = 6,
                match_prob: float = 0.7, target_std: float = 3.0, device="cpu") -> dict:
    """Greedy tree verification inputs: target ~ N(0, target_std^2) [B][N][V];
    the first child of every node holds the target's argmax after its parent
    with probability `match_prob` (else a uniform token), the other children
    uniform tokens; node 0's token is unused (0)."""
    g = _gen(seed, device)
    parent = tree_topology(branching)
    N = len(parent)
    target = _normal((B, N, V), target_std, g, device).to(dtype)
    best = torch.argmax(target.float(), dim=-1)
    rand_tok = torch.randint(0, V, (B, N), generator=g, device=device)
    keep = torch.rand((B, N), generator=g, device=device) < match_prob
    tokens = torch.zeros((B, N), dtype=torch.int64, device=device)
    first = {}
    for n in range(1, N):
        p = parent[n]
        is_first = p not in first
        first.setdefault(p, n)
        if is_first:
            tokens[:, n] = torch.where(keep[:, n], best[:, p], rand_tok[:, n])
        else:
            tokens[:, n] = rand_tok[:, n]
    par = torch.tensor(parent, dtype=torch.int32, device=device).expand(B, N).contiguous()
    return dict(name=f"tree greedy B={B} N={N} V={V} branching={tuple(branching)}", target=target,
                tree_tokens=tokens.to(torch.int32), parent=par, B=B, N=N, V=V)


def dynaspec_budget(kmax: int, K: int) -> list[int]:
    """Clusters drawn at draft step t = 0..K-1 under DynaSpec's position-aware
    budget (DynaSpec summary, § Method 3): kmax for t in {0, 1} and
    floor(kmax / ((t + 1) * 2)) for t >= 2, as printed, with at least one
    cluster, since an empty shortlist would leave the drafter nothing to
    propose.  Input generation only: the library never evaluates it."""
    return [kmax if t < 2 else max(1, kmax // ((t + 1) * 2)) for t in range(K)]


def shortlist_per_position(B: int = 64, K: int = 6, V: int = 262144, n_clusters: int = 64, budget=None,
                           dtype=torch.bfloat16, T: float = 1.0, sigma: float = 0.5, seed: int = 7,
                           device="cpu") -> dict:
    """Per-position shortlists: the vocabulary split at random into n_clusters
    clusters; at draft step t each sequence draws budget[t] clusters (default
    the DynaSpec position-aware budget with k_max = 8: 8, 8, 1, 1, 1, 1), whose
    sorted union is its list; target is full-vocabulary Zipf, the draft is
    target + N(0, sigma^2) on the list, compact [B][K][S] with S = max list
    length (row (b, t) holds len[t] entries); drafted tokens from the draft
    softmax on the list."""
    if budget is None:
        budget = dynaspec_budget(8, K)
    g = _gen(seed, device)
    target = zipf_logits(B * (K + 1), V, g, device).reshape(B, K + 1, V).to(dtype)
    size = V // n_clusters
    clusters = torch.randperm(V, generator=g, device=device)[:n_clusters * size].reshape(n_clusters, size)
    lens = [budget[t] * size for t in range(K)]
    S = max(lens)
    lists = torch.zeros((B, K, S), dtype=torch.int32, device=device)
    draft = torch.zeros((B, K, S), dtype=torch.float32, device=device)
    tokens = torch.zeros((B, K), dtype=torch.int32, device=device)
    for t in range(K):
        n = lens[t]
        for b in range(B):
            pick = torch.randperm(n_clusters, generator=g, device=device)[:budget[t]]
            lst = torch.sort(clusters[pick].reshape(-1)).values
            lists[b, t, :n] = lst.to(torch.int32)
        idx = lists[:, t, :n].long()
        draft[:, t, :n] = torch.gather(target[:, t].float(), 1, idx) + _normal((B, n), sigma, g, device)
        pos = gumbel_max_tokens(draft[:, t, :n].to(dtype), T, g).long()
        tokens[:, t] = torch.gather(idx, 1, pos[:, None])[:, 0].to(torch.int32)
    return dict(name=f"per-position shortlists B={B} K={K} V={V} lens={lens}", target=target,
                draft=draft.to(dtype), draft_tokens=tokens, T=T, shortlist=lists, shortlist_len=lens,
                B=B, K=K, V=V, S=S)
