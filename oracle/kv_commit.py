"""Oracle of the KV-cache commit / rollback that follows verification.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``).

What it computes (nextadmin.net lesson "Speculative Decoding", § KV cache
management): the verification pass feeds the K drafted tokens to the target
model in one forward pass, which extends its KV cache by K entries; when some
drafts are rejected, the cache must return to the length of the accepted
prefix.  Production systems write the K new entries to a staging buffer and
commit them once acceptance is known.  The same lesson's § Exercises, item 4,
fixes the outcome: a 10-token prefix, 5 drafts, a rejection at position 3 ->
the next iteration reads exactly the prefix plus the first 2 accepted drafts.

Readings (the pages leave these open):
  - the entries committed for sequence b are the first accept_len[b] staged
    entries (those of the accepted drafts); the token emitted at the
    rejection (or the bonus token) has no entry yet: it is the next round's
    input;
  - a negative accept_len (a sequence the verification reported in error)
    commits nothing;
  - a commit that would pass the cache's capacity L, or an accept_len above
    K, commits nothing and reports the sequence;
  - with no staging buffer (entries written in place at [len, len + K)), the
    commit is the length update alone: the rejected entries are rolled back
    by truncation.

Layout: cache [NL][B][L][W], staged [NL][B][K][W] (W bytes per entry and
layer, any element type), seq_len [B].
"""
from __future__ import annotations

import numpy as np

ERR_CAPACITY = 1


def kv_commit(cache, staged, seq_len, accept_len):
    """Returns (new cache, new seq_len, status [B]); the inputs are not modified."""
    cache = np.array(cache, copy=True)
    seq_len = np.array(seq_len, dtype=np.int64, copy=True)
    accept_len = np.asarray(accept_len, dtype=np.int64)
    B = seq_len.shape[0]
    L = cache.shape[2]
    K = staged.shape[2] if staged is not None else None
    status = np.zeros(B, dtype=np.int32)
    for b in range(B):
        a = int(accept_len[b])
        if a < 0:
            continue
        if (K is not None and a > K) or seq_len[b] + a > L:
            status[b] = ERR_CAPACITY
            continue
        n = int(seq_len[b])
        if staged is not None:
            cache[:, b, n:n + a] = staged[:, b, :a]
        seq_len[b] = n + a
    return cache, seq_len.astype(np.int32), status
