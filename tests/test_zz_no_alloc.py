"""spec_verify_static: verification with the library's own static scratch (no
workspace), for callers that cannot allocate device memory.  Collected last on
purpose: it must pass alone and after every other test, and the static scratch
must be left zeroed by the calls before, including one whose waits gave up."""
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


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(DEV)
    sv.load()


@pytest.fixture(autouse=True)
def _env():
    """spec_verify_static runs the cluster kernel; the workspace entry point is
    held to the same kernel, so the two calls compute the same sums."""
    keys = ("SPECVERIFY_KERNEL", "SPECVERIFY_SPIN_LIMIT")
    saved = {k: os.environ.get(k) for k in keys}
    os.environ["SPECVERIFY_KERNEL"] = "cluster"
    os.environ.pop("SPECVERIFY_SPIN_LIMIT", None)
    yield
    for k, v in saved.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = v


def _dev(cfg):
    return (cfg["target"].to(DEV), None if cfg["draft"] is None else cfg["draft"].to(DEV),
            cfg["draft_tokens"].to(DEV))


@pytest.mark.parametrize("which", ["stochastic", "greedy", "small_f32"])
def test_static_matches_workspace_entry_point_twice(which):
    if which == "stochastic":
        cfg = synth.throughput(B=64, K=4, seed=9)
    elif which == "greedy":
        cfg = synth.greedy(B=32, K=5, seed=7)
    else:
        cfg = synth.small_stochastic(seed=3)
    t, d, tok = _dev(cfg)
    T, seed = cfg["T"], 123
    if T == 0:
        ref_t, ref_l = sv.spec_verify_greedy(t, tok)
    else:
        ref_t, ref_l = sv.spec_verify(t, d, tok, T, seed)
    torch.cuda.synchronize()
    ref_t, ref_l = ref_t.cpu().numpy(), ref_l.cpu().numpy()
    for call in range(2):   # the scratch is left ready for the next call
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        got_t, got_l = sv.spec_verify_static(t, d, tok, T, seed, aux=sv.Aux(device_status=st))
        torch.cuda.synchronize()
        got_t, got_l = got_t.cpu().numpy(), got_l.cpu().numpy()
        # the same kernel (forced above) and the same uniforms: identical results
        np.testing.assert_array_equal(got_l, ref_l, err_msg=f"call {call}")
        np.testing.assert_array_equal(got_t, ref_t, err_msg=f"call {call}")
        assert int(st.cpu()[0]) == 0
    # and within the parity criterion of the oracle
    ref = oracle.verify(cfg["target"], cfg["draft"], cfg["draft_tokens"], T, seed)
    if T == 0:
        np.testing.assert_array_equal(got_t, ref["tokens"])
    else:
        assert_parity(got_t, got_l, ref, f"static {which}")


def test_static_rejects_shapes_that_need_a_workspace():
    cfg = synth.stochastic_gaussian(2, 2, 4097, torch.bfloat16, 1.0, 2.0, 0.5, seed=1)   # rows not 16-byte aligned
    t, d, tok = _dev(cfg)
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_verify_static(t, d, tok, 1.0, 1)
    assert e.value.code == 5   # SPEC_ERR_UNSUPPORTED
    aux = sv.Aux.alloc(2, 2, DEV)   # per-position outputs need the workspace kernel
    cfg = synth.stochastic_gaussian(2, 2, 4096, torch.bfloat16, 1.0, 2.0, 0.5, seed=1)
    t, d, tok = _dev(cfg)
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_verify_static(t, d, tok, 1.0, 1, aux=aux)
    assert e.value.code == 5


def test_static_after_waits_ran_out():
    """A call whose exchange waits gave up (spin limit 1: a CTA polls once for
    its peers' records) reports SPEC_ERR_TIMEOUT for the sequences it did not
    finish and leaves the static scratch zeroed: the next call, at the default
    limit, gives the oracle's results with status 0."""
    from test_gpu_timeout import check_gave_up
    cfg = synth.throughput(B=24, K=4, seed=13)
    t, d, tok = _dev(cfg)
    ref = oracle.verify(cfg["target"], cfg["draft"], cfg["draft_tokens"], 1.0, 31)
    os.environ["SPECVERIFY_SPIN_LIMIT"] = "1"
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    got_t, got_l = sv.spec_verify_static(t, d, tok, 1.0, 31, aux=sv.Aux(device_status=st))
    torch.cuda.synchronize()
    n = check_gave_up(got_t.cpu().numpy(), got_l.cpu().numpy(), int(st.cpu()[0]), ref, "static, spin limit 1")
    assert n > 0
    os.environ.pop("SPECVERIFY_SPIN_LIMIT")
    for call in range(2):
        st = torch.full((1,), -1, dtype=torch.int32, device=DEV)
        got_t, got_l = sv.spec_verify_static(t, d, tok, 1.0, 31, aux=sv.Aux(device_status=st))
        torch.cuda.synchronize()
        assert int(st.cpu()[0]) == 0
        assert_parity(got_t.cpu().numpy(), got_l.cpu().numpy(), ref, f"static after a timeout, call {call}")
