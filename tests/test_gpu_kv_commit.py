"""KV-cache commit (CUDA, through the C ABI) against its oracle: bit-exact
byte copies and lengths, on seeded inputs, including the page's rollback
exercise, in-place commits, ragged entry sizes and capacity errors."""
from __future__ import annotations

import json
import os

import numpy as np
import pytest
import torch

import speculative_decoding_verification_sampling_gb300 as sv
from oracle.kv_commit import kv_commit

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_rollback_exercise.json")


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(DEV)
    sv.load()


def _run(cache, staged, seq_len, acc, K=None):
    c = cache.to(DEV).contiguous()
    s = staged.to(DEV).contiguous() if staged is not None else None
    ln = torch.tensor(seq_len, dtype=torch.int32, device=DEV)
    st = torch.full((1,), -5, dtype=torch.int32, device=DEV)
    sv.spec_kv_commit(c, s, torch.tensor(acc, dtype=torch.int32, device=DEV), ln, K=K, device_status=st)
    return c.cpu(), ln.cpu().numpy(), int(st.item())


def _bytes(t):
    return t.contiguous().view(torch.uint8).numpy()


def test_rollback_exercise_from_the_page():
    g = json.load(open(GOLDEN))
    P, N = g["prefix_tokens"], g["drafted_tokens"]
    cache = torch.zeros((1, 1, 32, 8, 16), dtype=torch.bfloat16)
    cache[0, 0, :P] = torch.arange(1, P + 1, dtype=torch.bfloat16)[:, None, None]
    staged = torch.arange(100, 100 + N, dtype=torch.bfloat16)[None, None, :, None, None].expand(1, 1, N, 8, 16)
    c, ln, st = _run(cache, staged, [P], [g["accepted_drafts"]])
    assert ln[0] == g["cache_length_after"] and st == 0
    want = torch.cat([torch.arange(1, P + 1), torch.arange(100, 100 + g["accepted_drafts"])]).to(torch.bfloat16)
    assert torch.equal(c[0, 0, :ln[0], 0, 0], want)
    assert torch.equal(c[0, 0, ln[0]:], cache[0, 0, ln[0]:])


@pytest.mark.parametrize("NL,B,L,K,entry,dtype", [
    (3, 7, 40, 5, (8, 64), torch.bfloat16),    # 1 KB entries
    (2, 33, 70, 8, (2, 8, 128), torch.float16),
    (1, 5, 9, 4, (3,), torch.float32),         # 12-byte entries: the byte path
    (4, 64, 300, 6, (2, 8, 128), torch.bfloat16),
])
def test_commit_matches_oracle(NL, B, L, K, entry, dtype):
    g = torch.Generator().manual_seed(NL * 100 + B)
    cache = torch.randn((NL, B, L) + entry, generator=g).to(dtype)
    staged = torch.randn((NL, B, K) + entry, generator=g).to(dtype)
    seq_len = torch.randint(0, L + 1, (B,), generator=g).numpy()
    acc = torch.randint(-2, K + 2, (B,), generator=g).numpy()   # errors, overflows, K + 1
    c, ln, st = _run(cache, staged, seq_len, acc)
    oc, oln, ost = kv_commit(_bytes(cache).reshape(NL, B, L, -1), _bytes(staged).reshape(NL, B, K, -1), seq_len, acc)
    assert np.array_equal(_bytes(c).reshape(NL, B, L, -1), oc)
    assert np.array_equal(ln, oln)
    assert st == (1 if ost.any() else 0)


def test_in_place_commit():
    cache = torch.randn((2, 6, 20, 64), dtype=torch.float32)
    seq_len, acc = [0, 5, 19, 16, 10, 3], [4, 0, 1, 4, -1, 2]
    c, ln, st = _run(cache, None, seq_len, acc, K=4)
    oc, oln, ost = kv_commit(cache.numpy(), None, seq_len, acc)
    assert torch.equal(c, cache) and np.array_equal(ln, oln) and st == 0


def test_verify_then_commit():
    """The commit driven by a verification call's accept lengths."""
    from speculative_decoding_verification_sampling_gb300 import synth
    cfg = synth.stochastic_gaussian(16, 4, 5000, torch.bfloat16, 1.0, seed=3)
    t, l = sv.spec_verify(cfg["target"].to(DEV), cfg["draft"].to(DEV), cfg["draft_tokens"].to(DEV), 1.0, 11)
    cache = torch.zeros((2, 16, 64, 32), dtype=torch.bfloat16, device=DEV)
    staged = torch.randn((2, 16, 4, 32), device=DEV).to(torch.bfloat16)
    ln = torch.full((16,), 10, dtype=torch.int32, device=DEV)
    sv.spec_kv_commit(cache, staged, l, ln)
    lh = l.cpu()
    assert torch.equal(ln.cpu(), 10 + lh)
    for b in range(16):
        assert torch.equal(cache[:, b, 10:10 + lh[b]].cpu(), staged[:, b, :lh[b]].cpu())


def test_launch_count():
    cache = torch.zeros((1, 2, 8, 16), dtype=torch.uint8, device=DEV)
    staged = torch.ones((1, 2, 3, 16), dtype=torch.uint8, device=DEV)
    n0 = sv.spec_launch_count()
    sv.spec_kv_commit(cache, staged, torch.tensor([1, 2], dtype=torch.int32, device=DEV),
                      torch.tensor([0, 0], dtype=torch.int32, device=DEV))
    assert sv.spec_launch_count() == n0 + 2
