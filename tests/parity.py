"""Comparison of the CUDA path's outputs with the float64 oracle.

Greedy and error outputs must match exactly.  Sampled tokens must match
exactly except where the oracle reports a uniform within `band` (1e-6) of
its acceptance threshold min(1, q/p) at an examined position, or of a CDF
boundary of the distribution it sampled; such sequences are counted and
returned, never silently accepted.
"""
from __future__ import annotations

import numpy as np

BAND = 1e-6


def compare(gpu_tokens, gpu_len, ref, band: float = BAND):
    gt = np.asarray(gpu_tokens)
    gl = np.asarray(gpu_len)
    B, K1 = gt.shape
    K = K1 - 1
    bad, excused = [], []
    for b in range(B):
        if gl[b] == ref["accept_len"][b] and np.array_equal(gt[b], ref["tokens"][b]):
            continue
        term = int(ref["terminal"][b])
        near = False
        if term >= 0 and ref["accept_len"][b] >= 0 and gl[b] >= 0:
            upto = min(term, K - 1)
            near = bool((ref["accept_margin"][b, :upto + 1] < band).any()) or ref["sample_margin"][b] < band
        (excused if near else bad).append(b)
    return bad, excused


def assert_parity(gpu_tokens, gpu_len, ref, what: str, band: float = BAND, max_excused_frac: float = 0.01):
    bad, excused = compare(gpu_tokens, gpu_len, ref, band)
    n = len(ref["accept_len"])
    if bad:
        b = bad[0]
        raise AssertionError(
            f"{what}: {len(bad)} of {n} sequences differ from the oracle outside the {band} band; "
            f"first b={b}: gpu {np.asarray(gpu_tokens)[b].tolist()} len {int(np.asarray(gpu_len)[b])} | "
            f"oracle {ref['tokens'][b].tolist()} len {int(ref['accept_len'][b])} "
            f"margins {ref['accept_margin'][b].tolist()} / {ref['sample_margin'][b]}")
    assert len(excused) <= max(1, int(max_excused_frac * n)), f"{what}: {len(excused)} near-threshold"
    return len(excused)
