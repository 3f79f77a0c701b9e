"""spec_verify_static: verification with the library's own static scratch (no
workspace).  Collected last on purpose: it must pass alone and after every
other test, and the static scratch must be left zeroed by the calls before."""
from __future__ import annotations

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
        # same kernel, same uniforms: identical to the workspace entry point
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
