"""Float64 CPU oracle for batched speculative-decoding verification.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library in ``speculative_decoding_verification_sampling_gb300``,
and that library never calls it.

The arithmetic lives in ``oracle.c`` (plain C, float64), which cites the pages
it follows; this module only builds it with gcc and marshals numpy arrays.

Pinned by the ``-m "not gpu"`` tests in ``tests/test_oracle_pins.py``:
Philox against Triton's interpreter, the worked single-position example of the
runelab.ai post, brute-force enumeration on V <= 4, K <= 2, chi-square and
total-variation checks of the emitted distribution, the closed form for the
expected number of tokens per round, and special cases (p == q, one-hot q,
one-hot p, greedy against numpy.argmax); and, in ``tests/test_oracle_outputs.py``,
the per-position outputs and margins against scipy, and the tokens drawn for a
given seed: the accept decisions against u < min(1, q/p) evaluated by numpy and
the emitted token against numpy.searchsorted on the float64 CDF, both with the
uniforms rebuilt from the (Triton-pinned) Philox words.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (plain -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                               "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.oracle_philox4x32_10.argtypes = [P, P, P]
            lib.oracle_philox4x32_10.restype = None
            lib.oracle_uniform24.argtypes = [ctypes.c_uint32]
            lib.oracle_uniform24.restype = ctypes.c_double
            lib.oracle_softmax.argtypes = [P, ctypes.c_int, ctypes.c_double, P, P]
            lib.oracle_softmax.restype = ctypes.c_int
            lib.oracle_accept_prob.argtypes = [ctypes.c_double, ctypes.c_double]
            lib.oracle_accept_prob.restype = ctypes.c_double
            lib.oracle_residual.argtypes = [P, P, ctypes.c_int, P]
            lib.oracle_residual.restype = ctypes.c_double
            lib.oracle_inverse_cdf.argtypes = [P, ctypes.c_int, ctypes.c_double, ctypes.c_double, P]
            lib.oracle_inverse_cdf.restype = ctypes.c_int
            lib.oracle_argmax_first.argtypes = [P, ctypes.c_int]
            lib.oracle_argmax_first.restype = ctypes.c_int
            lib.oracle_verify.argtypes = [P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int,
                                          P, ctypes.c_int, P,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_double, ctypes.c_uint64,
                                          P, P, P, P, P, P, P, P, P, P, ctypes.c_int]
            lib.oracle_verify.restype = ctypes.c_int
            lib.oracle_verify_sl.argtypes = [P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int,
                                             P, ctypes.c_int, ctypes.c_longlong, ctypes.c_longlong, P, P,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_double, ctypes.c_uint64,
                                             P, P, P, P, P, P, P, P, P, P, ctypes.c_int]
            lib.oracle_verify_sl.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


# --------------------------------------------------------------------- steps
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform24(word: int) -> float:
    return _load().oracle_uniform24(int(word))


def softmax(z, T: float = 1.0):
    """Returns (probabilities, log-sum-exp) or raises ValueError on bad rows."""
    z = _f64(z)
    out = np.zeros_like(z)
    lse = ctypes.c_double()
    st = _load().oracle_softmax(_ptr(z), z.size, float(T), _ptr(out), ctypes.byref(lse))
    if st:
        raise ValueError("non-finite row")
    return out, lse.value


def accept_prob(q_d: float, p_d: float) -> float:
    return _load().oracle_accept_prob(float(q_d), float(p_d))


def residual(q, p):
    """Returns (r, R) with r = max(0, q - p) and R = sum(r)."""
    q, p = _f64(q), _f64(p)
    r = np.zeros_like(q)
    R = _load().oracle_residual(_ptr(q), _ptr(p), q.size, _ptr(r))
    return r, R


def inverse_cdf(r, R: float, v: float):
    """Returns (token, margin)."""
    r = _f64(r)
    m = ctypes.c_double()
    x = _load().oracle_inverse_cdf(_ptr(r), r.size, float(R), float(v), ctypes.byref(m))
    return x, m.value


def argmax_first(z) -> int:
    z = _f64(z)
    return _load().oracle_argmax_first(_ptr(z), z.size)


# --------------------------------------------------------------------- batch
def _raw(t):
    """A host array in the oracle's element codes: float32 as is, bfloat16 as its bits."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16), BF16
            if t.dtype == torch.float32:
                return t.numpy(), F32
            raise TypeError(f"unsupported dtype {t.dtype}")
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(t)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"unsupported dtype {a.dtype}")


def _i32(t):
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return np.ascontiguousarray(t.detach().cpu().to(torch.int32).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(t, dtype=np.int32))


def verify(target, draft, draft_tokens, T: float, seed: int, *, draft_is_probs: bool = False,
           shortlist=None, shortlist_len=None, full: bool = False, threads: int | None = None,
           seq_ids=None) -> dict:
    """One verification round for every sequence of the batch.

    target: [B][K+1][V] float32 or bfloat16 logits; draft: [B][K][V] logits or
    float32 probabilities ([B][K][S] with a ``shortlist``: [B][S] one list per
    sequence, [B][K][S] one list per position, or [S] one list shared by all;
    ``shortlist_len`` [K] the entries of each position's list, default S);
    draft_tokens: [B][K].  T == 0 selects greedy verification.  ``full`` also
    returns q_i(d_i), p_i(d_i) and the log-sum-exp of every row.
    Returns numpy arrays: tokens [B][K+1], accept_len [B], terminal [B],
    residual_mass [B], accept_margin [B][K], sample_margin [B] (and q_draft,
    p_draft, row_lse when ``full``).  ``seq_ids`` [B] gives the sequence index
    that keys each row's uniforms (default: the row number), so that a sample
    of a larger batch draws the same uniforms as the full batch.
    """
    tgt, tdt = _raw(target)
    B, K1, V = tgt.shape
    K = K1 - 1
    if T > 0:
        drf, ddt = _raw(draft)
        if draft_is_probs and ddt != F32:
            raise TypeError("draft probabilities must be float32")
    else:
        drf, ddt = None, F32
    tok = _i32(draft_tokens).reshape(B, K)
    sl = None
    S = 0
    sl_seq = sl_pos = 0
    sl_len = None
    if shortlist is not None:
        sl = _i32(shortlist)
        S = sl.shape[-1]
        if sl.ndim == 3:
            sl_seq, sl_pos = K * S, S
        elif sl.ndim == 2:
            sl_seq, sl_pos = S, 0
        if shortlist_len is not None:
            sl_len = np.ascontiguousarray(np.asarray(shortlist_len, dtype=np.int32))
    out_tokens = np.zeros((B, K + 1), dtype=np.int32)
    out_len = np.zeros(B, dtype=np.int32)
    terminal = np.zeros(B, dtype=np.int32)
    res_mass = np.zeros(B, dtype=np.float64)
    acc_margin = np.zeros((B, K), dtype=np.float64)
    smp_margin = np.zeros(B, dtype=np.float64)
    q_draft = p_draft = row_lse = None
    if full:
        q_draft = np.zeros((B, K), dtype=np.float64)
        p_draft = np.zeros((B, K), dtype=np.float64)
        row_lse = np.zeros((B, 2 * K + 1), dtype=np.float64)
    if threads is None:
        threads = os.cpu_count() or 1
    sid = None if seq_ids is None else np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int32))
    st = _load().oracle_verify_sl(_ptr(tgt), tdt, _ptr(drf), ddt, int(bool(draft_is_probs)),
                               _ptr(sl), S, sl_seq, sl_pos, _ptr(sl_len), _ptr(tok), B, K, V, float(T),
                               int(seed) & (2**64 - 1),
                               _ptr(out_tokens), _ptr(out_len), _ptr(q_draft), _ptr(p_draft),
                               _ptr(res_mass), _ptr(row_lse), _ptr(acc_margin), _ptr(smp_margin),
                               _ptr(terminal), _ptr(sid), int(threads))
    if st:
        raise ValueError("oracle_verify: invalid arguments")
    out = dict(tokens=out_tokens, accept_len=out_len, terminal=terminal, residual_mass=res_mass,
               accept_margin=acc_margin, sample_margin=smp_margin)
    if full:
        out.update(q_draft=q_draft, p_draft=p_draft, row_lse=row_lse)
    return out
