"""Batched speculative-decoding verification on GB300 (sm_103a).

A thin ctypes binding over ``libspecverify.so``, whose C ABI is declared in
``include/specverify.h``.  Every step of the verification runs in the
library's CUDA kernels; this module only checks tensor shapes and dtypes,
allocates outputs and scratch with PyTorch, and passes device pointers and
the current CUDA stream.  There is no CPU fallback: if the library is not
built, the calls raise.

Notation (nextadmin.net "Speculative Decoding", § Core algorithm): q is the
target distribution, p the draft distribution, d_i the K drafted tokens.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB as _LIB_PATH

__all__ = [
    "SpecVerifyError", "Aux", "spec_verify", "spec_verify_greedy", "spec_verify_shortlist",
    "spec_workspace_bytes", "spec_philox_words", "spec_draft_sample", "spec_kv_commit", "spec_verify_tree_greedy", "spec_tree_mask",
    "spec_verify_shortlist_pos", "spec_status_string", "spec_launch_count", "spec_verify_static", "library_path", "load",
]

SPEC_F32, SPEC_BF16 = 0, 1
STATUS = {0: "SPEC_OK", 1: "SPEC_ERR_INVALID_ARG", 2: "SPEC_ERR_NONFINITE", 3: "SPEC_ERR_TOKEN_RANGE",
          4: "SPEC_ERR_SHORTLIST", 5: "SPEC_ERR_UNSUPPORTED", 6: "SPEC_ERR_CUDA", 7: "SPEC_ERR_TIMEOUT"}


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)} ({spec_status_string(code)})")
        self.code = code


class _AuxStruct(ctypes.Structure):
    _fields_ = [("q_draft", ctypes.c_void_p), ("p_draft", ctypes.c_void_p),
                ("residual_mass", ctypes.c_void_p), ("row_lse", ctypes.c_void_p),
                ("device_status", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libspecverify.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise ImportError(f"{_LIB_PATH} is missing: build it first "
                                  "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(_LIB_PATH)
            P, I, U64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float
            Z = ctypes.c_size_t
            lib.spec_workspace_bytes.argtypes = [I, I, I, I]
            lib.spec_workspace_bytes.restype = Z
            lib.spec_verify.argtypes = [P, I, P, I, I, P, I, I, I, F, U64, P, P, P, Z, P, P]
            lib.spec_verify.restype = I
            lib.spec_verify_greedy.argtypes = [P, I, P, I, I, I, P, P, P, Z, P, P]
            lib.spec_verify_greedy.restype = I
            lib.spec_verify_shortlist.argtypes = [P, I, P, I, I, P, I, P, I, I, I, F, U64, P, P, P, Z, P, P]
            lib.spec_verify_shortlist.restype = I
            lib.spec_philox_words.argtypes = [U64, ctypes.c_uint32, I, I, P, P]
            lib.spec_philox_words.restype = I
            lib.spec_status_string.argtypes = [I]
            lib.spec_status_string.restype = ctypes.c_char_p
            lib.spec_verify_static.argtypes = [P, I, P, P, I, I, I, F, U64, P, P, P, P]
            lib.spec_verify_static.restype = I
            L64 = ctypes.c_longlong
            lib.spec_verify_shortlist_pos.argtypes = [P, I, P, I, P, L64, L64, P, I, P, I, I, I, F, U64, P, P, P,
                                                      Z, P, P]
            lib.spec_verify_shortlist_pos.restype = I
            lib.spec_tree_workspace_bytes.argtypes = [I, I, I]
            lib.spec_tree_workspace_bytes.restype = Z
            lib.spec_verify_tree_greedy.argtypes = [P, I, P, P, I, I, I, P, P, P, P, Z, P, P]
            lib.spec_verify_tree_greedy.restype = I
            lib.spec_tree_mask.argtypes = [P, I, I, P, P, P]
            lib.spec_tree_mask.restype = I
            lib.spec_kv_commit.argtypes = [P, P, I, I, I, I, Z, P, P, P, P]
            lib.spec_kv_commit.restype = I
            lib.spec_draft_sample.argtypes = [P, I, I, I, I, F, U64, P, P, P, P]
            lib.spec_draft_sample.restype = I
            lib.spec_launch_count.argtypes = []
            lib.spec_launch_count.restype = U64
            _lib = lib
    return _lib


def spec_launch_count() -> int:
    """Kernels the library has launched in this process (all entry points)."""
    return int(load().spec_launch_count())


def spec_status_string(code: int) -> str:
    return load().spec_status_string(int(code)).decode()


def spec_workspace_bytes(B: int, K: int, V: int, S: int = 0) -> int:
    return int(load().spec_workspace_bytes(int(B), int(K), int(V), int(S)))


class Aux:
    """Optional per-call outputs (device tensors, any may be None).  Asking for
    q_draft, p_draft or row_lse makes the call evaluate every position."""

    def __init__(self, q_draft=None, p_draft=None, residual_mass=None, row_lse=None, device_status=None):
        self.q_draft, self.p_draft, self.residual_mass = q_draft, p_draft, residual_mass
        self.row_lse, self.device_status = row_lse, device_status

    @classmethod
    def alloc(cls, B: int, K: int, device, full: bool = True) -> "Aux":
        f = dict(dtype=torch.float32, device=device)
        nan = float("nan")
        return cls(q_draft=torch.full((B, K), nan, **f) if full else None,
                   p_draft=torch.full((B, K), nan, **f) if full else None,
                   residual_mass=torch.full((B,), nan, **f),
                   row_lse=torch.full((B, 2 * K + 1), nan, **f) if full else None,
                   device_status=torch.full((1,), -1, dtype=torch.int32, device=device))

    def _struct(self, B, K):
        def ptr(t, shape, dtype):
            if t is None:
                return None
            _check(t, shape, (dtype,), "aux")
            return t.data_ptr()
        return _AuxStruct(ptr(self.q_draft, (B, K), torch.float32), ptr(self.p_draft, (B, K), torch.float32),
                          ptr(self.residual_mass, (B,), torch.float32),
                          ptr(self.row_lse, (B, 2 * K + 1), torch.float32),
                          ptr(self.device_status, (1,), torch.int32))


# ------------------------------------------------------------------ helpers
def _check(t, shape, dtypes, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dt(t):
    return SPEC_BF16 if t.dtype == torch.bfloat16 else SPEC_F32


_ws_cache: dict = {}


def _workspace(device, stream, nbytes, sizes):
    """A workspace cached per (device, stream).  The library leaves it ready
    for the next call with the same sizes; when the sizes change, it is
    zero-filled again (on the same stream) before the call."""
    key = (device.index, stream)
    ent = _ws_cache.get(key)
    if ent is None or ent[0].numel() < nbytes:
        ent = [torch.zeros(max(nbytes, 1 << 16), dtype=torch.uint8, device=device), sizes]
        _ws_cache[key] = ent
    elif ent[1] != sizes:
        ent[0].zero_()
        ent[1] = sizes
    return ent[0]


def _outs(B, K, device, out_tokens, out_accept_len):
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=device)
    if out_accept_len is None:
        out_accept_len = torch.empty((B,), dtype=torch.int32, device=device)
    _check(out_tokens, (B, K + 1), (torch.int32,), "out_tokens")
    _check(out_accept_len, (B,), (torch.int32,), "out_accept_len")
    return out_tokens, out_accept_len


def _stream(device, stream):
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ws_args(device, st, nbytes, workspace, sizes):
    if workspace is None:
        workspace = _workspace(device, st, nbytes, sizes)
    elif not isinstance(workspace, torch.Tensor) or not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA tensor")
    return workspace, workspace.numel() * workspace.element_size()


# ------------------------------------------------------------------ entry points
def spec_verify(target: torch.Tensor, draft: torch.Tensor, draft_tokens: torch.Tensor, T: float, seed: int,
                *, draft_is_probs: bool = False, out_tokens=None, out_accept_len=None, workspace=None,
                aux: Aux | None = None, stream=None):
    """One verification round for B sequences.

    target [B][K+1][V] float32/bfloat16 logits; draft [B][K][V] logits of the
    same dtype, or float32 probabilities with ``draft_is_probs``; draft_tokens
    [B][K] int32.  T == 0 runs the greedy rule.  Returns (out_tokens [B][K+1],
    out_accept_len [B]) on the device, asynchronously on the current stream.
    """
    B, K1, V = target.shape
    K = K1 - 1
    _check(target, (B, K + 1, V), (torch.float32, torch.bfloat16), "target")
    _check(draft, (B, K, V), (torch.float32,) if draft_is_probs else (target.dtype,), "draft")
    _check(draft_tokens, (B, K), (torch.int32,), "draft_tokens")
    dev = target.device
    out_tokens, out_accept_len = _outs(B, K, dev, out_tokens, out_accept_len)
    st = _stream(dev, stream)
    workspace, wsb = _ws_args(dev, st, spec_workspace_bytes(B, K, V, 0), workspace, (B, K, V, 0))
    ax = aux._struct(B, K) if aux is not None else None
    rc = load().spec_verify(target.data_ptr(), _dt(target), draft.data_ptr(), _dt(draft), int(draft_is_probs),
                            draft_tokens.data_ptr(), B, K, V, float(T), int(seed) & (2**64 - 1),
                            out_tokens.data_ptr(), out_accept_len.data_ptr(), workspace.data_ptr(), wsb,
                            ctypes.byref(ax) if ax is not None else None, st)
    if rc:
        raise SpecVerifyError(rc, "spec_verify")
    return out_tokens, out_accept_len


def spec_verify_greedy(target: torch.Tensor, draft_tokens: torch.Tensor, *, out_tokens=None,
                       out_accept_len=None, workspace=None, aux: Aux | None = None, stream=None):
    """Greedy verification: accept d_i while d_i == argmax q_i (lowest index on ties)."""
    B, K1, V = target.shape
    K = K1 - 1
    _check(target, (B, K + 1, V), (torch.float32, torch.bfloat16), "target")
    _check(draft_tokens, (B, K), (torch.int32,), "draft_tokens")
    dev = target.device
    out_tokens, out_accept_len = _outs(B, K, dev, out_tokens, out_accept_len)
    st = _stream(dev, stream)
    workspace, wsb = _ws_args(dev, st, spec_workspace_bytes(B, K, V, 0), workspace, (B, K, V, 0))
    ax = aux._struct(B, K) if aux is not None else None
    rc = load().spec_verify_greedy(target.data_ptr(), _dt(target), draft_tokens.data_ptr(), B, K, V,
                                   out_tokens.data_ptr(), out_accept_len.data_ptr(), workspace.data_ptr(), wsb,
                                   ctypes.byref(ax) if ax is not None else None, st)
    if rc:
        raise SpecVerifyError(rc, "spec_verify_greedy")
    return out_tokens, out_accept_len


def spec_verify_static(target: torch.Tensor, draft: torch.Tensor | None, draft_tokens: torch.Tensor, T: float,
                       seed: int, *, out_tokens=None, out_accept_len=None, aux: Aux | None = None, stream=None):
    """spec_verify without a workspace: the library's own 256-byte scratch
    (see include/specverify.h).  Draft logits only; T == 0 is greedy (draft
    may be None).  Raises SpecVerifyError (SPEC_ERR_UNSUPPORTED) for shapes
    that need a workspace.  Calls must not overlap on the GPU."""
    B, K1, V = target.shape
    K = K1 - 1
    _check(target, (B, K + 1, V), (torch.float32, torch.bfloat16), "target")
    if T > 0:
        _check(draft, (B, K, V), (target.dtype,), "draft")
    _check(draft_tokens, (B, K), (torch.int32,), "draft_tokens")
    dev = target.device
    out_tokens, out_accept_len = _outs(B, K, dev, out_tokens, out_accept_len)
    st = _stream(dev, stream)
    ax = aux._struct(B, K) if aux is not None else None
    rc = load().spec_verify_static(target.data_ptr(), _dt(target), draft.data_ptr() if (draft is not None and T > 0)
                                   else None, draft_tokens.data_ptr(), B, K, V, float(T), int(seed),
                                   out_tokens.data_ptr(), out_accept_len.data_ptr(),
                                   ctypes.byref(ax) if ax is not None else None, st)
    if rc:
        raise SpecVerifyError(rc, "spec_verify_static")
    return out_tokens, out_accept_len


def spec_verify_shortlist(target: torch.Tensor, draft_sl: torch.Tensor, shortlist_idx: torch.Tensor,
                          draft_tokens: torch.Tensor, T: float, seed: int, *, draft_is_probs: bool = False,
                          out_tokens=None, out_accept_len=None, workspace=None, aux: Aux | None = None,
                          stream=None):
    """Verification with a draft defined on a per-sequence shortlist.

    draft_sl [B][K][S] (logits of the target's dtype, or float32 probabilities),
    shortlist_idx [B][S] int32 strictly ascending inside [0, V)."""
    B, K1, V = target.shape
    K = K1 - 1
    S = shortlist_idx.shape[-1]
    _check(target, (B, K + 1, V), (torch.float32, torch.bfloat16), "target")
    _check(draft_sl, (B, K, S), (torch.float32,) if draft_is_probs else (target.dtype,), "draft_sl")
    _check(shortlist_idx, (B, S), (torch.int32,), "shortlist_idx")
    _check(draft_tokens, (B, K), (torch.int32,), "draft_tokens")
    dev = target.device
    out_tokens, out_accept_len = _outs(B, K, dev, out_tokens, out_accept_len)
    st = _stream(dev, stream)
    workspace, wsb = _ws_args(dev, st, spec_workspace_bytes(B, K, V, S), workspace, (B, K, V, S))
    ax = aux._struct(B, K) if aux is not None else None
    rc = load().spec_verify_shortlist(target.data_ptr(), _dt(target), draft_sl.data_ptr(), _dt(draft_sl),
                                      int(draft_is_probs), shortlist_idx.data_ptr(), S, draft_tokens.data_ptr(),
                                      B, K, V, float(T), int(seed) & (2**64 - 1), out_tokens.data_ptr(),
                                      out_accept_len.data_ptr(), workspace.data_ptr(), wsb,
                                      ctypes.byref(ax) if ax is not None else None, st)
    if rc:
        raise SpecVerifyError(rc, "spec_verify_shortlist")
    return out_tokens, out_accept_len


def spec_philox_words(seed: int, tag: int, B: int, P: int, device=None, stream=None) -> torch.Tensor:
    """The Philox4x32-10 words the kernels draw: [B][P][4] (int32 storage of uint32)."""
    device = torch.device(device if device is not None else "cuda")
    out = torch.empty((B, P, 4), dtype=torch.int32, device=device)
    st = _stream(device, stream)
    rc = load().spec_philox_words(int(seed) & (2**64 - 1), int(tag), B, P, out.data_ptr(), st)
    if rc:
        raise SpecVerifyError(rc, "spec_philox_words")
    return out


def spec_draft_sample(draft: torch.Tensor, T: float, seed: int, *, out_tokens=None, out_prob=None,
                      device_status=None, stream=None):
    """Draft tokens d_i ~ softmax(draft[b][i] / T) by inverse CDF on Philox
    uniforms (counter (i, b, 1, 0)), with p_i(d_i).  draft [B][K][V] float32 or
    bfloat16 logits.  T == 0 takes the first argmax (probability 1).  Returns
    (out_tokens [B][K] int32, out_prob [B][K] float32) on the device."""
    B, K, V = draft.shape
    _check(draft, (B, K, V), (torch.float32, torch.bfloat16), "draft")
    dev = draft.device
    if out_tokens is None:
        out_tokens = torch.empty((B, K), dtype=torch.int32, device=dev)
    if out_prob is None:
        out_prob = torch.empty((B, K), dtype=torch.float32, device=dev)
    _check(out_tokens, (B, K), (torch.int32,), "out_tokens")
    _check(out_prob, (B, K), (torch.float32,), "out_prob")
    if device_status is not None:
        _check(device_status, (1,), (torch.int32,), "device_status")
    st = _stream(dev, stream)
    rc = load().spec_draft_sample(draft.data_ptr(), _dt(draft), B, K, V, float(T), int(seed) & (2**64 - 1),
                                  out_tokens.data_ptr(), out_prob.data_ptr(),
                                  device_status.data_ptr() if device_status is not None else None, st)
    if rc:
        raise SpecVerifyError(rc, "spec_draft_sample")
    return out_tokens, out_prob


def spec_kv_commit(cache: torch.Tensor, staged: torch.Tensor | None, accept_len: torch.Tensor,
                   seq_len: torch.Tensor, *, K: int | None = None, device_status=None, stream=None):
    """Commit the accepted drafts' KV entries: cache [NL][B][L][...] (any
    dtype), staged [NL][B][K][...] of the same dtype and entry shape (None:
    entries written in place, then K must be given), accept_len [B] int32 (as
    spec_verify returns it), seq_len [B] int32 updated in place."""
    if not isinstance(cache, torch.Tensor) or not cache.is_cuda or cache.dim() < 4 or not cache.is_contiguous():
        raise TypeError("cache must be a contiguous CUDA tensor [NL][B][L][...]")
    NL, B, L = cache.shape[:3]
    entry = cache[0, 0, 0]
    W = entry.numel() * cache.element_size()
    if staged is not None:
        K = staged.shape[2]
        _check(staged, (NL, B, K) + tuple(cache.shape[3:]), (cache.dtype,), "staged")
    elif K is None:
        raise ValueError("K is needed when the entries were written in place")
    _check(accept_len, (B,), (torch.int32,), "accept_len")
    _check(seq_len, (B,), (torch.int32,), "seq_len")
    if device_status is not None:
        _check(device_status, (1,), (torch.int32,), "device_status")
    st = _stream(cache.device, stream)
    rc = load().spec_kv_commit(cache.data_ptr(), staged.data_ptr() if staged is not None else None, NL, B, int(K), L,
                               W, accept_len.data_ptr(), seq_len.data_ptr(),
                               device_status.data_ptr() if device_status is not None else None, st)
    if rc:
        raise SpecVerifyError(rc, "spec_kv_commit")
    return seq_len


def spec_verify_tree_greedy(target: torch.Tensor, tree_tokens: torch.Tensor, parent: torch.Tensor, *,
                            workspace=None, device_status=None, stream=None):
    """Greedy verification of a draft tree: target [B][N][V] logits (row n: the
    prediction after node n), tree_tokens and parent [B][N] int32 (parent[0]
    == -1, parent[n] < n).  Returns (out_tokens [B][N], out_nodes [B][N],
    out_accept_len [B])."""
    B, N, V = target.shape
    _check(target, (B, N, V), (torch.float32, torch.bfloat16), "target")
    _check(tree_tokens, (B, N), (torch.int32,), "tree_tokens")
    _check(parent, (B, N), (torch.int32,), "parent")
    dev = target.device
    nbytes = int(load().spec_tree_workspace_bytes(B, N, V))
    if nbytes == 0:
        raise SpecVerifyError(1, "spec_verify_tree_greedy")
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out_t = torch.empty((B, N), dtype=torch.int32, device=dev)
    out_n = torch.empty((B, N), dtype=torch.int32, device=dev)
    out_l = torch.empty((B,), dtype=torch.int32, device=dev)
    if device_status is not None:
        _check(device_status, (1,), (torch.int32,), "device_status")
    st = _stream(dev, stream)
    rc = load().spec_verify_tree_greedy(target.data_ptr(), _dt(target), tree_tokens.data_ptr(), parent.data_ptr(),
                                        B, N, V, out_t.data_ptr(), out_n.data_ptr(), out_l.data_ptr(),
                                        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                        device_status.data_ptr() if device_status is not None else None, st)
    if rc:
        raise SpecVerifyError(rc, "spec_verify_tree_greedy")
    return out_t, out_n, out_l


def spec_tree_mask(parent: torch.Tensor, *, out=None, device_status=None, stream=None) -> torch.Tensor:
    """Tree attention mask: uint8 [B][N][N], 1 where node j is node i or an ancestor of it."""
    B, N = parent.shape
    _check(parent, (B, N), (torch.int32,), "parent")
    if out is None:
        out = torch.empty((B, N, N), dtype=torch.uint8, device=parent.device)
    _check(out, (B, N, N), (torch.uint8,), "out")
    if device_status is not None:
        _check(device_status, (1,), (torch.int32,), "device_status")
    rc = load().spec_tree_mask(parent.data_ptr(), B, N, out.data_ptr(),
                               device_status.data_ptr() if device_status is not None else None,
                               _stream(parent.device, stream))
    if rc:
        raise SpecVerifyError(rc, "spec_tree_mask")
    return out


def spec_verify_shortlist_pos(target: torch.Tensor, draft_sl: torch.Tensor, shortlist_idx: torch.Tensor,
                              draft_tokens: torch.Tensor, T: float, seed: int, *, shortlist_len=None,
                              out_tokens=None, out_accept_len=None, workspace=None, aux: Aux | None = None,
                              stream=None):
    """Verification with per-position shortlists: shortlist_idx [B][K][S] (one
    list per position), [B][S] (one per sequence) or [S] (one shared list), int32
    strictly ascending; draft_sl [B][K][S] logits of the target's dtype, row
    (b, i) holding shortlist_len[i] entries (a host sequence of K ints; default S)."""
    B, K1, V = target.shape
    K = K1 - 1
    S = shortlist_idx.shape[-1]
    _check(target, (B, K + 1, V), (torch.float32, torch.bfloat16), "target")
    _check(draft_sl, (B, K, S), (target.dtype,), "draft_sl")
    _check(draft_tokens, (B, K), (torch.int32,), "draft_tokens")
    if shortlist_idx.dim() == 3:
        _check(shortlist_idx, (B, K, S), (torch.int32,), "shortlist_idx")
        seq, pos = K * S, S
    elif shortlist_idx.dim() == 2:
        _check(shortlist_idx, (B, S), (torch.int32,), "shortlist_idx")
        seq, pos = S, 0
    else:
        _check(shortlist_idx, (S,), (torch.int32,), "shortlist_idx")
        seq, pos = 0, 0
    lens = None
    if shortlist_len is not None:
        lens = (ctypes.c_int32 * K)(*[int(x) for x in shortlist_len])
    dev = target.device
    out_tokens, out_accept_len = _outs(B, K, dev, out_tokens, out_accept_len)
    st = _stream(dev, stream)
    workspace, wsb = _ws_args(dev, st, spec_workspace_bytes(B, K, V, S), workspace, (B, K, V, S))
    ax = aux._struct(B, K) if aux is not None else None
    rc = load().spec_verify_shortlist_pos(target.data_ptr(), _dt(target), draft_sl.data_ptr(), _dt(draft_sl),
                                          shortlist_idx.data_ptr(), seq, pos, lens, S, draft_tokens.data_ptr(),
                                          B, K, V, float(T), int(seed) & (2**64 - 1), out_tokens.data_ptr(),
                                          out_accept_len.data_ptr(), workspace.data_ptr(), wsb,
                                          ctypes.byref(ax) if ax is not None else None, st)
    if rc:
        raise SpecVerifyError(rc, "spec_verify_shortlist_pos")
    return out_tokens, out_accept_len
