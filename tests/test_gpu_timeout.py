"""Timeout paths of the kernels, made to run out without a GPU fault.

Every wait on another CTA is bounded by the spin limit (SPECVERIFY_SPIN_LIMIT);
waits on a CTA's own barriers (its copies, its hand-offs between warps) keep a
floor that the limit does not lower, so a CTA never winds down with its own
copies still landing.  At a spin limit of 1 the waits on other CTAs give up at
once unless what they wait for is already there:

- the row-parallel statistics stream: its producers' wait for every sequence
  to have ended, and for a posted residual job to be written;
- the resident kernel for small calls: each CTA's wait for its sequence's end;
- the cluster kernel: the exchange of per-CTA records inside a cluster;
- the chunk-scheduled kernel: an idle worker's wait for its residual slot.

A sequence whose outputs were not finished reports SPEC_ERR_TIMEOUT (7) with
every token -1; the others must still be the oracle's.  The device status is
7 exactly when a sequence timed out.  The next call, at the default limit, must
give the oracle's results with status 0: the context is usable and the call's
control words were left zeroed.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_sampling_gb300 as sv
from parity import assert_parity
from speculative_decoding_verification_sampling_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TIMEOUT = 7
KEYS = ("SPECVERIFY_KERNEL", "SPECVERIFY_ROWS_FUSED", "SPECVERIFY_SPIN_LIMIT", "SPECVERIFY_ROWS_RESIDENT")


@pytest.fixture(autouse=True)
def _env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    saved = {k: os.environ.get(k) for k in KEYS}
    yield
    for k, v in saved.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = v


def _run(cfg, seed, aux=None):
    t, l = sv.spec_verify(cfg["target"].to(DEV), cfg["draft"].to(DEV), cfg["draft_tokens"].to(DEV), cfg["T"],
                          seed, aux=aux)
    torch.cuda.synchronize()
    return t.cpu().numpy(), l.cpu().numpy()


def check_gave_up(t, l, status, ref, what):
    """Sequences that timed out carry -7 and -1 tokens; the rest are the
    oracle's; the status is 7 exactly when one timed out."""
    out = l == -TIMEOUT
    assert (t[out] == -1).all(), what
    assert status == (TIMEOUT if out.any() else 0), (what, status, int(out.sum()))
    keep = ~out
    if keep.any():
        sub = {k: v[keep] for k, v in ref.items()}
        assert_parity(t[keep], l[keep], sub, what)
    return int(out.sum())


def run_out_then_recover(cfg, seed, what, must_time_out=True, all_out=False):
    ref = oracle.verify(cfg["target"], cfg["draft"], cfg["draft_tokens"], cfg["T"], seed)
    os.environ["SPECVERIFY_SPIN_LIMIT"] = "1"
    aux = sv.Aux(device_status=torch.zeros(1, dtype=torch.int32, device=DEV))
    t, l = _run(cfg, seed, aux=aux)
    n = check_gave_up(t, l, int(aux.device_status.cpu()[0]), ref, what + " (spin limit 1)")
    if must_time_out:
        assert n > 0, f"{what}: no wait ran out at spin limit 1"
    if all_out:
        assert n == len(l), f"{what}: {n} of {len(l)} sequences timed out"
    os.environ.pop("SPECVERIFY_SPIN_LIMIT")
    aux = sv.Aux(device_status=torch.full((1,), -1, dtype=torch.int32, device=DEV))
    t, l = _run(cfg, seed, aux=aux)
    assert int(aux.device_status.cpu()[0]) == 0
    assert_parity(t, l, ref, f"{what}, after a timeout")


@pytest.mark.parametrize("B,K", [(64, 4), (256, 4)])
def test_stream_waits_run_out_then_recover(B, K):
    """The stream's producers give up at once: every sequence reports 7."""
    os.environ["SPECVERIFY_KERNEL"] = "rows"
    os.environ["SPECVERIFY_ROWS_FUSED"] = "1"
    run_out_then_recover(synth.throughput(B=B, K=K, seed=B + 7), 5, f"stream B={B} K={K}", all_out=True)


@pytest.mark.parametrize("B,K", [(1, 4), (8, 4)])
def test_resident_waits_run_out_then_recover(B, K):
    """The resident kernel's CTAs wait for their sequence's end; at spin limit
    1 those that commit before it is known give up, and every sequence
    reports 7."""
    os.environ["SPECVERIFY_ROWS_RESIDENT"] = "1"
    run_out_then_recover(synth.throughput(B=B, K=K, seed=B + 9), 6, f"resident B={B} K={K}", all_out=True)


@pytest.mark.parametrize("B,K,V", [(24, 4, 128256), (16, 3, 8192)])
def test_cluster_exchange_waits_run_out_then_recover(B, K, V):
    os.environ["SPECVERIFY_KERNEL"] = "cluster"
    cfg = synth.stochastic_gaussian(B, K, V, torch.bfloat16, 1.0, 2.0, 0.5, seed=B + V)
    run_out_then_recover(cfg, 8, f"cluster B={B} K={K} V={V}")


@pytest.mark.parametrize("B,K,V", [(48, 4, 16384), (8, 5, 3000)])
def test_general_kernel_waits_run_out_then_recover(B, K, V):
    os.environ["SPECVERIFY_KERNEL"] = "general"
    cfg = synth.stochastic_gaussian(B, K, V, torch.bfloat16, 1.0, 2.0, 0.5, seed=B + V)
    run_out_then_recover(cfg, 9, f"chunk-scheduled B={B} K={K} V={V}")
