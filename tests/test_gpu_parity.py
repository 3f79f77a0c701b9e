"""CUDA path against the float64 oracle, through the C ABI, on seeded synthetic
inputs: greedy bit-exact; sampled tokens identical except near-threshold
uniforms (counted); probabilities within 1e-5 absolute."""
from __future__ import annotations

import math
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


@pytest.fixture(scope="module", autouse=True,
                params=["auto", "cluster", "rows", "rows-stats", "rows-unfused", "general"])
def kernel(request):
    """Every case runs under the default dispatch (small aligned calls: the
    resident kernel) and under each kernel forced in turn: the cluster kernel,
    the row-parallel kernels
    (with the bulk-copy statistics stream, and with the per-position
    statistics launches in its place: "rows-stats") and the chunk-scheduled
    kernel (each falls back to the next for shapes it does not serve);
    "rows" runs the residual pass inside the statistics stream at every size,
    "rows-unfused" keeps it in its own launch and runs greedy calls on the
    register-load argmax kernel even where rows are aligned for bulk copies."""
    keys = ("SPECVERIFY_KERNEL", "SPECVERIFY_ROWS_STREAM", "SPECVERIFY_ROWS_FUSED", "SPECVERIFY_GREEDY_CFG",
            "SPECVERIFY_ROWS_RESIDENT")
    saved = {k: os.environ.get(k) for k in keys}
    os.environ["SPECVERIFY_KERNEL"] = "rows" if request.param.startswith("rows") else request.param
    if request.param == "rows-stats":
        os.environ["SPECVERIFY_ROWS_STREAM"] = "0"
    if request.param == "rows":
        os.environ["SPECVERIFY_ROWS_FUSED"] = "1"
        os.environ["SPECVERIFY_ROWS_RESIDENT"] = "0"
    if request.param == "rows-unfused":
        os.environ["SPECVERIFY_ROWS_FUSED"] = "0"
        os.environ["SPECVERIFY_ROWS_RESIDENT"] = "0"
        os.environ["SPECVERIFY_GREEDY_CFG"] = "256,2"
    yield request.param
    for k, v in saved.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = v


def _to(cfg):
    out = {}
    for k in ("target", "draft", "draft_tokens", "shortlist"):
        v = cfg.get(k)
        out[k] = None if v is None else v.to(DEV).contiguous()
    return out


def _gpu_run(cfg, seed, aux=None, probs=False):
    d = _to(cfg)
    if cfg.get("shortlist") is not None:
        t, l = sv.spec_verify_shortlist(d["target"], d["draft"], d["shortlist"], d["draft_tokens"], cfg["T"],
                                        seed, draft_is_probs=probs, aux=aux)
    elif cfg["T"] == 0:
        t, l = sv.spec_verify_greedy(d["target"], d["draft_tokens"], aux=aux)
    else:
        t, l = sv.spec_verify(d["target"], d["draft"], d["draft_tokens"], cfg["T"], seed, draft_is_probs=probs,
                              aux=aux)
    torch.cuda.synchronize()
    return t.cpu().numpy(), l.cpu().numpy()


def _oracle(cfg, seed, idx=None, full=False, probs=False):
    sel = (lambda x: x) if idx is None else (lambda x: None if x is None else x[idx])
    return oracle.verify(sel(cfg["target"]), sel(cfg["draft"]), sel(cfg["draft_tokens"]), cfg["T"], seed,
                         shortlist=sel(cfg.get("shortlist")), full=full, draft_is_probs=probs,
                         seq_ids=None if idx is None else np.asarray(idx, dtype=np.int32))


# ------------------------------------------------------------------ Philox
def test_philox_words_match_oracle():
    B, P = 37, 33
    for seed in (0, 1234567, 0xDEADBEEFCAFEF00D):
        got = sv.spec_philox_words(seed, 0, B, P, DEV).cpu().numpy().view(np.uint32)
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for b in range(0, B, 5):
            for p in range(0, P, 4):
                want = oracle.philox4x32_10([p, b, 0, 0], key)
                np.testing.assert_array_equal(got[b, p], want)


# ------------------------------------------------------------------ greedy
def test_greedy_full_size_bit_exact():
    cfg = synth.greedy()                       # B=64, K=5, V=128256 bf16
    t, l = _gpu_run(cfg, 0)
    ref = _oracle(cfg, 0)
    np.testing.assert_array_equal(l, ref["accept_len"])
    np.testing.assert_array_equal(t, ref["tokens"])


@pytest.mark.parametrize("B,K,V,dtype", [
    (1, 1, 1, torch.float32), (3, 31, 257, torch.float32), (5, 7, 4097, torch.bfloat16),
    (2, 3, 50257, torch.bfloat16), (16, 4, 1000, torch.float32), (9, 2, 8192 * 3 + 8, torch.bfloat16),
    (4, 3, 16, torch.float32), (7, 4, 300, torch.float32), (40, 2, 128256, torch.bfloat16),
])
def test_greedy_edge_shapes(B, K, V, dtype):
    cfg = synth.greedy(B=B, K=K, V=V, dtype=dtype, seed=B * 100 + K)
    t, l = _gpu_run(cfg, 0)
    ref = _oracle(cfg, 0)
    np.testing.assert_array_equal(l, ref["accept_len"])
    np.testing.assert_array_equal(t, ref["tokens"])


@pytest.mark.parametrize("B,K,V,dtype", [
    (96, 3, 32768, torch.bfloat16),    # 2.5 rows per SM, rows of exactly four copy stages
    (48, 7, 16388, torch.float32),     # a last stage of 16 bytes
    (256, 5, 40000, torch.bfloat16),   # several waves of CTAs
])
def test_greedy_many_rows(B, K, V, dtype):
    """Many aligned rows of 64 KB or more run on the bulk-copy kernel, one CTA
    per row (the "rows-unfused" pass runs them on the register-load kernel)."""
    cfg = _cached(("gm", B, K, V), lambda: synth.greedy(B=B, K=K, V=V, dtype=dtype, seed=B + V))
    ref = _cached(("gm-ref", B, K, V), lambda: _oracle(cfg, 0))
    t, l = _gpu_run(cfg, 0)
    np.testing.assert_array_equal(l, ref["accept_len"])
    np.testing.assert_array_equal(t, ref["tokens"])


@pytest.mark.parametrize("B,V", [(40, 20000), (64, 40000)])
def test_greedy_heavy_ties_across_parts(B, V):
    """Integer logits in [-2, 2]: the maximum appears in many parts of a row
    (B=40: several parts per row; B=64: one CTA per row, many warps); the
    lowest index must win."""
    g = torch.Generator().manual_seed(6)
    K = 5
    target = torch.randint(-2, 3, (B, K + 1, V), generator=g).to(torch.bfloat16)
    target[:, :, :V // 2] = torch.clamp(target[:, :, :V // 2], max=1)   # the first 2s sit past the middle
    best = torch.argmax(target[:, :K].float(), dim=-1)
    tokens = torch.where(torch.rand(B, K, generator=g) < 0.8, best, torch.randint(0, V, (B, K), generator=g))
    cfg = dict(target=target, draft=None, draft_tokens=tokens.to(torch.int32), T=0.0)
    t, l = _gpu_run(cfg, 0)
    ref = _oracle(cfg, 0)
    np.testing.assert_array_equal(l, ref["accept_len"])
    np.testing.assert_array_equal(t, ref["tokens"])


def test_greedy_heavy_ties():
    g = torch.Generator().manual_seed(5)
    B, K, V = 24, 6, 3000
    target = torch.randint(-2, 3, (B, K + 1, V), generator=g).to(torch.bfloat16)
    best = torch.argmax(target[:, :K].float(), dim=-1)
    tokens = torch.where(torch.rand(B, K, generator=g) < 0.8, best, torch.randint(0, V, (B, K), generator=g))
    cfg = dict(target=target, draft=None, draft_tokens=tokens.to(torch.int32), T=0.0)
    t, l = _gpu_run(cfg, 0)
    ref = _oracle(cfg, 0)
    np.testing.assert_array_equal(l, ref["accept_len"])
    np.testing.assert_array_equal(t, ref["tokens"])


# ------------------------------------------------------------------ stochastic
def test_small_fp32_config_many_seeds():
    cfg = synth.small_stochastic()              # B=1, K=4, V=32000 f32
    excused = 0
    for seed in range(40):
        t, l = _gpu_run(cfg, seed)
        excused += assert_parity(t, l, _oracle(cfg, seed), f"small seed {seed}")
    assert excused <= 1


@pytest.mark.parametrize("sigma", [0.25, 0.5, 1.0])
def test_zipf_config(sigma):
    cfg = synth.zipf(sigma=sigma)               # B=32, K=7, V=152064 bf16, T=0.7
    for seed in (1, 2):
        t, l = _gpu_run(cfg, seed)
        assert_parity(t, l, _oracle(cfg, seed), f"zipf sigma={sigma} seed={seed}")


@pytest.mark.parametrize("B,K", [(1, 4), (8, 4), (64, 4), (1, 8), (8, 8), (64, 8)])
def test_throughput_points_full(B, K):
    cfg = synth.throughput(B=B, K=K, seed=B + K)
    t, l = _gpu_run(cfg, 77)
    assert_parity(t, l, _oracle(cfg, 77), f"throughput B={B} K={K}")


# inputs and oracle results of the large cases, made once for every kernel
_CACHE = {}


def _cached(key, make):
    if key not in _CACHE:
        _CACHE[key] = make()
    return _CACHE[key]


@pytest.mark.parametrize("B,K", [(256, 4), (512, 8)])
def test_throughput_points_full_size(B, K):
    """The headline sizes, every sequence checked against the oracle."""
    cfg = _cached(("tp", B, K), lambda: synth.throughput(B=B, K=K, seed=B + K))
    ref = _cached(("tp-ref", B, K), lambda: _oracle(cfg, 99))
    t, l = _gpu_run(cfg, 99)
    assert_parity(t, l, ref, f"throughput B={B} K={K}")
    assert ((l >= 0) & (l <= K)).all()


def _sparse_rows(B, K, V, seed):
    """Target and draft rows that are -inf except on a few tokens (down to a
    single one), with drafted tokens on the draft's support, off it (p(d) = 0:
    accepted), and where the target is -inf (q(d) = 0)."""
    g = torch.Generator().manual_seed(seed)
    tgt = torch.full((B, K + 1, V), -math.inf)
    drf = torch.full((B, K, V), -math.inf)
    tok = torch.zeros((B, K), dtype=torch.int32)
    sizes = [1, 1, 2, 3, 5, 40, 300]
    for b in range(B):
        for i in range(K + 1):
            n = sizes[(b + i) % len(sizes)]
            sup = torch.randperm(V, generator=g)[:n]
            tgt[b, i, sup] = 2.0 * torch.randn(n, generator=g)
            if i == K:
                continue
            kind = (b * 7 + i) % 5
            if kind == 1:      # a single token, most likely off the target's support
                dsup = torch.randperm(V, generator=g)[:1]
            elif kind == 2:    # part of the target's support
                dsup = sup[:max(1, n // 2)]
            elif kind == 3:    # the target's support and a few tokens more
                dsup = torch.cat([sup, torch.randperm(V, generator=g)[:3]])
            elif kind == 4:    # somewhere else
                dsup = torch.randperm(V, generator=g)[:sizes[(b + 2 * i) % len(sizes)]]
            else:              # the target's support
                dsup = sup
            vals = torch.where(torch.isfinite(tgt[b, i, dsup]), tgt[b, i, dsup], torch.zeros(len(dsup)))
            drf[b, i, dsup] = vals + 0.5 * torch.randn(len(dsup), generator=g)
            both = torch.nonzero(torch.isfinite(drf[b, i]) & torch.isfinite(tgt[b, i]))[:, 0]
            fin = both if len(both) else torch.nonzero(torch.isfinite(drf[b, i]))[:, 0]
            pick = int(fin[torch.randint(len(fin), (1,), generator=g)])
            if (b + i) % 6 == 5:   # off the draft's support: p(d) = 0, accepted
                pick = int(torch.randint(V, (1,), generator=g))
            tok[b, i] = pick
    return dict(target=tgt.to(torch.bfloat16), draft=drf.to(torch.bfloat16), draft_tokens=tok, T=1.0)


@pytest.mark.parametrize("B,K,V", [(32, 4, 65536), (6, 3, 4096)])
def test_mostly_minus_inf_rows(B, K, V):
    cfg = _cached(("sparse", B, K, V), lambda: _sparse_rows(B, K, V, seed=B + V))
    for seed in (1, 2, 3):
        ref = _oracle(cfg, seed)
        assert (ref["accept_len"] >= 0).all()
        t, l = _gpu_run(cfg, seed)
        assert_parity(t, l, ref, f"mostly -inf rows B={B} V={V} seed={seed}")


def test_shortlist_config_full_vocabulary_form():
    """The shortlisted-draft workload in the form the DynaSpec summary states
    (§ Abstract: the drafter works on the shortlist, verification keeps the
    full vocabulary): B=64, K=6, V=262144, the draft a full-vocabulary row that
    is -inf off each sequence's 32,768-token shortlist.  spec_verify on that
    form matches the oracle and the compact spec_verify_shortlist call."""
    cfg = _cached("sl", synth.shortlist)
    B, K, V = cfg["B"], cfg["K"], cfg["V"]

    def full_form():
        full = torch.full((B, K, V), -math.inf, dtype=torch.bfloat16)
        full.scatter_(2, cfg["shortlist"].long().unsqueeze(1).expand(B, K, -1), cfg["draft"])
        return dict(target=cfg["target"], draft=full, draft_tokens=cfg["draft_tokens"], T=cfg["T"])

    fcfg = _cached("sl-full", full_form)
    ref = _cached("sl-full-ref", lambda: _oracle(fcfg, 21))
    t, l = _gpu_run(fcfg, 21)
    assert_parity(t, l, ref, "shortlist workload, full-vocabulary draft")
    ct, cl = _gpu_run(cfg, 21)
    assert_parity(ct, cl, ref, "shortlist workload, compact draft")
    np.testing.assert_array_equal(l, cl)
    np.testing.assert_array_equal(t, ct)


@pytest.mark.parametrize("B,K,V,dtype,T", [
    (3, 1, 1, torch.float32, 1.0), (4, 31, 300, torch.float32, 0.9), (7, 5, 4097, torch.bfloat16, 1.3),
    (5, 3, 50257, torch.bfloat16, 1.0), (2, 6, 2049, torch.float32, 0.5), (33, 2, 8192 * 2 + 16, torch.bfloat16, 1.0),
    (5, 3, 16, torch.float32, 1.0), (6, 4, 1004, torch.float32, 0.8), (300, 3, 2048, torch.bfloat16, 1.0),
])
def test_stochastic_edge_shapes(B, K, V, dtype, T):
    cfg = synth.stochastic_gaussian(B, K, V, dtype, T, 2.0, 0.5, seed=B * 7 + K)
    for seed in (3, 4):
        t, l = _gpu_run(cfg, seed)
        assert_parity(t, l, _oracle(cfg, seed), f"edge B={B} K={K} V={V}")


def test_misaligned_rows_take_the_direct_path():
    """A view starting one element into its storage is not 16-byte aligned."""
    B, K, V = 6, 3, 4096
    cfg = synth.stochastic_gaussian(B, K, V, torch.bfloat16, 1.0, 2.0, 0.5, seed=8)
    big_t = torch.empty(B * (K + 1) * V + 1, dtype=torch.bfloat16, device=DEV)
    big_d = torch.empty(B * K * V + 1, dtype=torch.bfloat16, device=DEV)
    tgt = big_t[1:].view(B, K + 1, V)
    drf = big_d[1:].view(B, K, V)
    tgt.copy_(cfg["target"])
    drf.copy_(cfg["draft"])
    t, l = sv.spec_verify(tgt, drf, cfg["draft_tokens"].to(DEV), 1.0, 5)
    torch.cuda.synchronize()
    assert_parity(t.cpu().numpy(), l.cpu().numpy(), _oracle(cfg, 5), "misaligned")


# ------------------------------------------------------------------ shortlist
def test_shortlist_full_size():
    cfg = synth.shortlist()                     # B=64, K=6, V=262144, S=32768
    t, l = _gpu_run(cfg, 21)
    assert_parity(t, l, _oracle(cfg, 21), "shortlist")


@pytest.mark.parametrize("B,K,V,S,dtype", [
    (4, 3, 1000, 37, torch.float32), (6, 5, 5000, 1000, torch.bfloat16), (3, 2, 600, 600, torch.bfloat16),
])
def test_shortlist_edge_shapes(B, K, V, S, dtype):
    g = torch.Generator().manual_seed(V + S)
    target = (2.0 * torch.randn(B, K + 1, V, generator=g)).to(dtype)
    sl = torch.stack([torch.sort(torch.randperm(V, generator=g)[:S]).values for _ in range(B)]).to(torch.int32)
    draft = (torch.gather(target[:, :K].float(), 2, sl.long().unsqueeze(1).expand(B, K, S))
             + 0.5 * torch.randn(B, K, S, generator=g)).to(dtype)
    pos = synth.gumbel_max_tokens(draft, 1.0, g).long()
    tok = torch.gather(sl.long(), 1, pos).to(torch.int32)
    tok[0, 0] = int((set(range(V)) - set(sl[0].tolist())).pop()) if S < V else tok[0, 0]   # off-shortlist draft
    cfg = dict(target=target, draft=draft, draft_tokens=tok, T=1.0, shortlist=sl)
    for seed in (1, 2, 3):
        t, l = _gpu_run(cfg, seed)
        assert_parity(t, l, _oracle(cfg, seed), f"shortlist edge V={V} S={S}")


# ------------------------------------------------------------------ probabilities
@pytest.mark.parametrize("B,K,V,dtype", [(32, 4, 5000, torch.float32), (16, 3, 12345, torch.bfloat16)])
def test_draft_probabilities(B, K, V, dtype):
    cfg = synth.stochastic_gaussian(B, K, V, dtype, 1.0, 2.0, 0.7, seed=V)
    probs = torch.softmax(cfg["draft"].double(), dim=-1).float()
    pc = dict(cfg, draft=probs)
    for seed in (5, 6):
        t, l = _gpu_run(pc, seed, probs=True)
        assert_parity(t, l, _oracle(pc, seed, probs=True), "probs")


def test_draft_probabilities_throughput_size():
    """Draft probabilities at B=256 K=4 V=128256 (the row-parallel path reads
    the target rows and, at each sequence's end, its probability row)."""
    cfg = _cached(("tp", 256, 4), lambda: synth.throughput(B=256, K=4, seed=260))
    pc = _cached(("tp-probs", 256, 4), lambda: dict(cfg, draft=torch.softmax(cfg["draft"].float(), dim=-1)))
    ref = _cached(("tp-probs-ref", 256, 4), lambda: _oracle(pc, 17, probs=True))
    t, l = _gpu_run(pc, 17, probs=True)
    assert_parity(t, l, ref, "draft probabilities B=256 K=4")


def test_draft_probability_errors_where_read():
    """Bad given probabilities are errors only where the rule reads them: the
    drafted token's p_i(d_i) at an examined position, and the whole row p_j at
    a rejection (its residual); an entry elsewhere in an accepted row is never
    read.  64 sequences of each kind, so the call takes the row-parallel path."""
    B, K, V = 256, 2, 4096
    q = torch.full((V,), 1.0 / V)
    tgt = torch.log(q).expand(B, K + 1, V).contiguous()
    drf = q.expand(B, K, V).contiguous().clone()
    tok = torch.zeros((B, K), dtype=torch.int32)
    for b in range(0, B, 4):
        drf[b, 0, 5] = -0.25            # p == q at the drafted token: accepted, entry 5 never read
        drf[b + 1, 0, 0] = math.nan     # the drafted token's own probability
        drf[b + 2, 0, 0] = 2.0 / V      # q/p = 0.5: some seeds reject, then the row is read
        drf[b + 2, 0, 3] = math.inf
        drf[b + 3, 1, 7] = -1.0         # position 1 row: read if position 1 rejects
        drf[b + 3, 1, 0] = 4.0 / V
    cfg = dict(target=tgt, draft=drf, draft_tokens=tok, T=1.0)
    for seed in (2, 3):
        ref = _oracle(cfg, seed, probs=True)
        t, l = _gpu_run(cfg, seed, probs=True)
        np.testing.assert_array_equal(l, ref["accept_len"])
        np.testing.assert_array_equal(t, ref["tokens"])
        assert (ref["accept_len"][0::4] == K).all() and (ref["accept_len"][1::4] == -2).all()
        assert -2 in ref["accept_len"][2::4] and (ref["accept_len"][2::4] != -2).any()


# ------------------------------------------------------------------ per-position outputs
@pytest.mark.parametrize("kind", ["logits", "probs", "shortlist"])
def test_per_position_outputs(kind):
    B, K, V = 24, 5, 7000
    cfg = synth.stochastic_gaussian(B, K, V, torch.bfloat16, 0.8, 2.0, 0.5, seed=31)
    probs = False
    if kind == "probs":
        cfg = dict(cfg, draft=torch.softmax(cfg["draft"].double() / 0.8, dim=-1).float())
        probs = True
    if kind == "shortlist":
        g = torch.Generator().manual_seed(3)
        S = 900
        sl = torch.stack([torch.sort(torch.randperm(V, generator=g)[:S]).values for _ in range(B)]).to(torch.int32)
        draft = torch.gather(cfg["draft"].float(), 2, sl.long().unsqueeze(1).expand(B, K, S)).to(torch.bfloat16)
        tok = torch.gather(sl.long(), 1, synth.gumbel_max_tokens(draft, 0.8, g).long()).to(torch.int32)
        cfg = dict(cfg, draft=draft, draft_tokens=tok, shortlist=sl)
    aux = sv.Aux.alloc(B, K, DEV)
    t, l = _gpu_run(cfg, 13, aux=aux, probs=probs)
    ref = _oracle(cfg, 13, full=True, probs=probs)
    assert_parity(t, l, ref, f"aux {kind}")
    q, p = aux.q_draft.cpu().numpy(), aux.p_draft.cpu().numpy()
    np.testing.assert_array_equal(np.isnan(q), np.isnan(ref["q_draft"]))
    np.testing.assert_allclose(q, ref["q_draft"], atol=1e-5, rtol=0)
    np.testing.assert_allclose(p, ref["p_draft"], atol=1e-5, rtol=0)
    lse = aux.row_lse.cpu().numpy()
    np.testing.assert_array_equal(np.isnan(lse), np.isnan(ref["row_lse"]))
    np.testing.assert_allclose(lse, ref["row_lse"], atol=1e-5, rtol=1e-6)
    ok = ~np.isnan(ref["residual_mass"])
    np.testing.assert_allclose(aux.residual_mass.cpu().numpy()[ok], ref["residual_mass"][ok], atol=1e-5, rtol=0)
    assert int(aux.device_status.cpu()[0]) == 0


# ------------------------------------------------------------------ data errors
def test_data_errors_per_sequence():
    B, K, V = 8, 3, 600
    cfg = synth.stochastic_gaussian(B, K, V, torch.float32, 1.0, 2.0, 0.0, seed=4)   # draft == target
    tgt, drf, tok = cfg["target"].clone(), cfg["draft"].clone(), cfg["draft_tokens"].clone()
    tgt[0, 0, 3] = math.nan
    tgt[1, 0, :] = -math.inf
    tok[2, 0] = V
    drf[3, 0, 5] = math.inf
    tgt[4, K, 1] = math.nan       # bonus row: reached because draft == target
    tok[5, 1] = -1
    tgt[6, K - 1, 0] = math.inf
    c = dict(cfg, target=tgt, draft=drf, draft_tokens=tok)
    aux = sv.Aux(device_status=torch.zeros(1, dtype=torch.int32, device=DEV))
    t, l = _gpu_run(c, 1, aux=aux)
    ref = _oracle(c, 1)
    np.testing.assert_array_equal(l, ref["accept_len"])
    np.testing.assert_array_equal(t, ref["tokens"])
    assert list(l[:7]) == [-2, -2, -3, -2, -2, -3, -2] and l[7] == K
    assert int(aux.device_status.cpu()[0]) in (2, 3)


def test_greedy_and_shortlist_errors():
    cfg = synth.greedy(B=4, K=3, V=900, dtype=torch.float32, seed=3)
    tgt = cfg["target"].clone()
    tgt[1, 0, 10] = math.nan
    tok = cfg["draft_tokens"].clone()
    tok[2, 0] = 900
    c = dict(cfg, target=tgt, draft_tokens=tok)
    t, l = _gpu_run(c, 0)
    ref = _oracle(c, 0)
    np.testing.assert_array_equal(l, ref["accept_len"])
    np.testing.assert_array_equal(t, ref["tokens"])
    g = torch.Generator().manual_seed(1)
    B, K, V, S = 3, 2, 500, 40
    target = torch.randn(B, K + 1, V, generator=g)
    sl = torch.stack([torch.sort(torch.randperm(V, generator=g)[:S]).values for _ in range(B)]).to(torch.int32)
    sl[1, 5] = sl[1, 4]           # duplicate
    sl[2, 0] = -3                 # out of range
    draft = torch.randn(B, K, S, generator=g)
    tok = sl[:, :K].clone()
    sc = dict(target=target, draft=draft, draft_tokens=tok, T=1.0, shortlist=sl)
    t, l = _gpu_run(sc, 2)
    ref = _oracle(sc, 2)
    np.testing.assert_array_equal(l, ref["accept_len"])
    assert list(l[1:]) == [-4, -4]


# ------------------------------------------------------------------ behaviour
def test_deterministic_and_workspace_left_zeroed():
    cfg = synth.throughput(B=64, K=4, seed=3)
    d = _to(cfg)
    B, K, V = 64, 4, 128256
    ws = torch.zeros(sv.spec_workspace_bytes(B, K, V), dtype=torch.uint8, device=DEV)
    outs = []
    for _ in range(3):
        t, l = sv.spec_verify(d["target"], d["draft"], d["draft_tokens"], 1.0, 42, workspace=ws)
        torch.cuda.synchronize()
        outs.append((t.cpu().numpy(), l.cpu().numpy()))
        # the control words a call must find zeroed are zero again
        assert int(ws[:256].count_nonzero()) == 0
    for t, l in outs[1:]:
        np.testing.assert_array_equal(t, outs[0][0])
        np.testing.assert_array_equal(l, outs[0][1])


def test_greedy_workspace_reused_across_batches():
    """Greedy calls on one workspace, alternating two batches: each matches the
    oracle, so every counter a call uses is back at zero for the next."""
    B, K, V = 48, 5, 20000
    cfgs = [synth.greedy(B=B, K=K, V=V, seed=s) for s in (41, 42)]
    refs = [_oracle(c, 0) for c in cfgs]
    ws = torch.zeros(sv.spec_workspace_bytes(B, K, V), dtype=torch.uint8, device=DEV)
    dev = [_to(c) for c in cfgs]
    for call in range(4):
        d, ref = dev[call % 2], refs[call % 2]
        st = torch.full((1,), -1, dtype=torch.int32, device=DEV)
        t, l = sv.spec_verify_greedy(d["target"], d["draft_tokens"], workspace=ws,
                                     aux=sv.Aux(device_status=st))
        torch.cuda.synchronize()
        np.testing.assert_array_equal(l.cpu().numpy(), ref["accept_len"])
        np.testing.assert_array_equal(t.cpu().numpy(), ref["tokens"])
        assert int(st.cpu()[0]) == 0
        assert int(ws[:256].count_nonzero()) == 0


def test_gpu_output_distribution_chi_square():
    """Exercise: the speculative histogram matches the target distribution
    (chi-square) -- here on the GPU with 100,000 sequences at V=8."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(3)
    V, K, B = 8, 3, 100_000
    zt = rng.normal(0, 1.5, size=(K + 1, V))
    zd = zt[:K] + rng.normal(0, 0.8, size=(K, V))
    pd = np.exp(zd - zd.max(-1, keepdims=True))
    pd /= pd.sum(-1, keepdims=True)
    tokens = np.stack([rng.choice(V, size=B, p=pd[i]) for i in range(K)], axis=1).astype(np.int32)
    tgt = torch.tensor(zt, dtype=torch.float32, device=DEV).unsqueeze(0).expand(B, -1, -1).contiguous()
    drf = torch.tensor(zd, dtype=torch.float32, device=DEV).unsqueeze(0).expand(B, -1, -1).contiguous()
    t, l = sv.spec_verify(tgt, drf, torch.tensor(tokens, device=DEV), 1.0, 2024)
    first = t[:, 0].cpu().numpy()
    q1 = np.exp(zt[0] - zt[0].max())
    q1 /= q1.sum()
    assert chisquare(np.bincount(first, minlength=V), q1 * B).pvalue > 1e-3


# ------------------------------------------------------------------ every output slot written
POISON = 0x7F7F7F7F


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_outputs_fully_written_over_poison(T):
    """Outputs pre-filled with 0x7F7F7F7F: every slot is written (unused token
    slots as -1), and the results are the oracle's."""
    B, K, V = 32, 4, 4096
    cfg = synth.stochastic_gaussian(B, K, V, torch.bfloat16, T if T > 0 else 1.0, 2.0, 0.5, seed=21)
    cfg = dict(cfg, T=T)
    d = _to(cfg)
    ot = torch.full((B, K + 1), POISON, dtype=torch.int32, device=DEV)
    ol = torch.full((B,), POISON, dtype=torch.int32, device=DEV)
    if T == 0:
        sv.spec_verify_greedy(d["target"], d["draft_tokens"], out_tokens=ot, out_accept_len=ol)
    else:
        sv.spec_verify(d["target"], d["draft"], d["draft_tokens"], T, 9, out_tokens=ot, out_accept_len=ol)
    torch.cuda.synchronize()
    t, l = ot.cpu().numpy(), ol.cpu().numpy()
    assert not (t == POISON).any() and not (l == POISON).any()
    assert_parity(t, l, _oracle(cfg, 9), f"poisoned outputs T={T}")
