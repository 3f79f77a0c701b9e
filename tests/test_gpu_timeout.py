"""The timeout path of the row-parallel statistics stream, made to run out
without a GPU fault.

With the spin limit at 1, the stream's producers give up at once on their
waits on other CTAs: for every sequence to have ended, and for a posted
residual job to be written. A producer that gives up sets the timeout word,
stops claiming work and still closes its ring, so the CTA drains every copy it
issued before it exits. Waits on the CTA's own barriers keep a floor that
the spin limit does not lower.

The call must report SPEC_ERR_TIMEOUT (7) for every sequence and in the
device status. The next call, at the default limit, must give the oracle's
results: the context is usable and the call's counters were left zeroed.
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


@pytest.fixture(autouse=True)
def _env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    keys = ("SPECVERIFY_KERNEL", "SPECVERIFY_ROWS_FUSED", "SPECVERIFY_SPIN_LIMIT")
    saved = {k: os.environ.get(k) for k in keys}
    os.environ["SPECVERIFY_KERNEL"] = "rows"
    os.environ["SPECVERIFY_ROWS_FUSED"] = "1"
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


@pytest.mark.parametrize("B,K", [(64, 4), (256, 4)])
def test_stream_waits_run_out_then_recover(B, K):
    cfg = synth.throughput(B=B, K=K, seed=B + 7)
    os.environ["SPECVERIFY_SPIN_LIMIT"] = "1"
    aux = sv.Aux(device_status=torch.zeros(1, dtype=torch.int32, device=DEV))
    t, l = _run(cfg, 5, aux=aux)
    assert int(aux.device_status.cpu()[0]) == TIMEOUT
    assert (l == -TIMEOUT).all()
    assert (t == -1).all()

    os.environ.pop("SPECVERIFY_SPIN_LIMIT")
    aux = sv.Aux(device_status=torch.full((1,), -1, dtype=torch.int32, device=DEV))
    t, l = _run(cfg, 5, aux=aux)
    assert int(aux.device_status.cpu()[0]) == 0
    assert_parity(t, l, oracle.verify(cfg["target"], cfg["draft"], cfg["draft_tokens"], cfg["T"], 5),
                  f"after a timeout, B={B} K={K}")
