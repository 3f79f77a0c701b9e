"""The C-ABI library builds, loads and exports every symbol that
include/specverify.h declares; host-side argument checks (no GPU needed)."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

import speculative_decoding_verification_sampling_gb300 as sv
from speculative_decoding_verification_sampling_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_]+)\s*\(", text)))


def test_library_builds_and_loads():
    path = lib_build.build()
    assert os.path.exists(path)
    assert sv.load() is not None


def test_every_declared_symbol_is_exported():
    decl = _declared()
    assert {"spec_verify", "spec_verify_greedy", "spec_verify_shortlist", "spec_workspace_bytes",
            "spec_status_string", "spec_philox_words"} <= set(decl)
    out = subprocess.run(["nm", "-D", "--defined-only", lib_build.build()], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (spec_[a-z_]+)\b", out))
    assert set(decl) <= exported, set(decl) - exported


def test_launch_counter_does_not_count_rejected_calls():
    lib = sv.load()
    n0 = sv.spec_launch_count()
    buf = (ctypes.c_int32 * 64)()
    p = ctypes.cast(buf, ctypes.c_void_p)
    assert lib.spec_verify(p, 0, p, 0, 0, p, 0, 4, 16, 1.0, 1, p, p, p, 1 << 8, None, None) == 1
    assert sv.spec_launch_count() == n0


def test_status_strings():
    for code in range(8):
        assert sv.spec_status_string(code)
    assert "wait" in sv.spec_status_string(7)


def test_workspace_bytes():
    a = sv.spec_workspace_bytes(256, 4, 128256)
    b = sv.spec_workspace_bytes(256, 4, 128256, 32768)
    assert 0 < a < 64 << 20 and 0 < b < 64 << 20
    # a smaller shortlist needs no more workspace than a larger one
    assert sv.spec_workspace_bytes(256, 4, 128256, 1024) <= b
    assert sv.spec_workspace_bytes(0, 4, 100) == 0
    assert sv.spec_workspace_bytes(1, 32, 100) == 0        # K above 31
    assert sv.spec_workspace_bytes(1, 0, 100) == 0
    assert sv.spec_workspace_bytes(1, 4, 100, 101) == 0    # S above V
    assert sv.spec_workspace_bytes(4096, 31, 262144) > 0


def test_invalid_arguments_return_before_any_launch():
    lib = sv.load()
    buf = (ctypes.c_int32 * 64)()
    ws = ctypes.create_string_buffer(1 << 20)
    p = ctypes.cast(buf, ctypes.c_void_p)
    w = ctypes.cast(ws, ctypes.c_void_p)
    # B = 0
    assert lib.spec_verify(p, 0, p, 0, 0, p, 0, 4, 16, 1.0, 1, p, p, w, 1 << 20, None, None) == 1
    # K = 32
    assert lib.spec_verify(p, 0, p, 0, 0, p, 1, 32, 16, 1.0, 1, p, p, w, 1 << 20, None, None) == 1
    # negative / NaN temperature
    assert lib.spec_verify(p, 0, p, 0, 0, p, 1, 4, 16, -1.0, 1, p, p, w, 1 << 20, None, None) == 1
    assert lib.spec_verify(p, 0, p, 0, 0, p, 1, 4, 16, float("nan"), 1, p, p, w, 1 << 20, None, None) == 1
    # draft probabilities must be float32; draft logits must match the target dtype
    assert lib.spec_verify(p, 1, p, 1, 1, p, 1, 4, 16, 1.0, 1, p, p, w, 1 << 20, None, None) == 1
    assert lib.spec_verify(p, 1, p, 0, 0, p, 1, 4, 16, 1.0, 1, p, p, w, 1 << 20, None, None) == 1
    # missing draft / workspace / too small workspace
    assert lib.spec_verify(p, 0, None, 0, 0, p, 1, 4, 16, 1.0, 1, p, p, w, 1 << 20, None, None) == 1
    assert lib.spec_verify(p, 0, p, 0, 0, p, 1, 4, 16, 1.0, 1, p, p, None, 1 << 20, None, None) == 1
    assert lib.spec_verify(p, 0, p, 0, 0, p, 1, 4, 16, 1.0, 1, p, p, w, 64, None, None) == 1
    # shortlist: S < 1, S > V, missing index
    assert lib.spec_verify_shortlist(p, 0, p, 0, 0, p, 0, p, 1, 4, 16, 1.0, 1, p, p, w, 1 << 20, None, None) == 1
    assert lib.spec_verify_shortlist(p, 0, p, 0, 0, p, 17, p, 1, 4, 16, 1.0, 1, p, p, w, 1 << 20, None, None) == 1
    assert lib.spec_verify_shortlist(p, 0, p, 0, 0, None, 8, p, 1, 4, 16, 1.0, 1, p, p, w, 1 << 20, None, None) == 1
    # greedy: bad dtype
    assert lib.spec_verify_greedy(p, 5, p, 1, 4, 16, p, p, w, 1 << 20, None, None) == 1
    assert lib.spec_philox_words(1, 0, 0, 4, p, None) == 1


def test_binding_rejects_cpu_tensors():
    import torch
    t = torch.zeros(1, 5, 16)
    with pytest.raises(TypeError):
        sv.spec_verify(t, t[:, :4].contiguous(), torch.zeros(1, 4, dtype=torch.int32), 1.0, 0)


def test_draft_sample_rejects_bad_arguments():
    """Argument errors come back before anything is launched."""
    lib = sv.load()
    p = ctypes.c_void_p(256)
    n0 = sv.spec_launch_count()
    assert lib.spec_draft_sample(None, 1, 1, 1, 8, 1.0, 0, p, None, None, None) == 1
    assert lib.spec_draft_sample(p, 1, 0, 1, 8, 1.0, 0, p, None, None, None) == 1
    assert lib.spec_draft_sample(p, 1, 1, 0, 8, 1.0, 0, p, None, None, None) == 1
    assert lib.spec_draft_sample(p, 1, 1, 1, 0, 1.0, 0, p, None, None, None) == 1
    assert lib.spec_draft_sample(p, 1, 1, 1, 8, -1.0, 0, p, None, None, None) == 1
    assert lib.spec_draft_sample(p, 1, 1, 1, 8, float("nan"), 0, p, None, None, None) == 1
    assert lib.spec_draft_sample(p, 1, 1, 1, 8, float("inf"), 0, p, None, None, None) == 1
    assert lib.spec_draft_sample(p, 7, 1, 1, 8, 1.0, 0, p, None, None, None) == 1
    assert lib.spec_draft_sample(p, 1, 1, 1, 1 << 22, 1.0, 0, p, None, None, None) == 5
    assert sv.spec_launch_count() == n0


def test_kv_commit_rejects_bad_arguments():
    lib = sv.load()
    p = ctypes.c_void_p(256)
    n0 = sv.spec_launch_count()
    assert lib.spec_kv_commit(None, p, 1, 1, 1, 1, 16, p, p, None, None) == 1
    assert lib.spec_kv_commit(p, p, 0, 1, 1, 1, 16, p, p, None, None) == 1
    assert lib.spec_kv_commit(p, p, 1, 0, 1, 1, 16, p, p, None, None) == 1
    assert lib.spec_kv_commit(p, p, 1, 1, 0, 1, 16, p, p, None, None) == 1
    assert lib.spec_kv_commit(p, p, 1, 1, 1, 0, 16, p, p, None, None) == 1
    assert lib.spec_kv_commit(p, p, 1, 1, 1, 1, 0, p, p, None, None) == 1
    assert lib.spec_kv_commit(p, p, 1, 1, 1, 1, 16, None, p, None, None) == 1
    assert lib.spec_kv_commit(p, p, 1, 1, 1, 1, 16, p, None, None, None) == 1
    assert lib.spec_kv_commit(p, p, 1 << 20, 1 << 20, 1, 1 << 20, 1 << 20, p, p, None, None) == 1
    assert sv.spec_launch_count() == n0
