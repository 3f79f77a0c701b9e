#!/usr/bin/env python3
"""Throughput of batched speculative-decoding verification on one GB300.

One step is one `spec_verify` call (the whole path: temperature softmax
statistics, left-to-right accept/reject, residual or bonus sampling) over the
throughput workload: B=256 sequences, K=4 drafted tokens, V=128256, bf16
target and draft logits, T=1, target logits ~ N(0, 2^2) and draft logits =
target + N(0, 0.5^2), drafted tokens sampled from the draft softmax.

Metric: verified draft positions per second (B*K per step).  Inputs live in
HBM when the timed region starts; each step reads one of `--rotate` device
copies of the 591 MB input set, so every step starts with the L2 (129 MB)
holding none of its rows.  Timing: `--warmup` untimed steps, then exactly
`--steps` steps between a barrier and a device synchronize on both sides,
timed with CUDA events on the launching stream; the maximum over ranks is
reported.  With N > 1 (torchrun, one process per GPU) every rank verifies its
own independent batch (replicas; nothing is exchanged).

Besides the device-timed value the JSON line carries:
  e2e          - the same metric through the public call with host buffers:
                 every step copies its inputs from pinned host memory and
                 reads its outputs back;
  roofline     - HBM roofline of the verification call (its four kernels,
                 timed together with CUDA events around each call): the logits
                 the left-to-right rule must read (rows up to the first
                 rejection, or all 2K+1 rows when every draft is accepted) over
                 the mean call duration, against the measured copy bandwidth;
                 `traffic` is the DRAM bytes of all four kernels of one call;
  cpu_baseline - the float64 CPU oracle on this host's cores, on a bounded
                 sample of the same batch (rank 0, one GPU only);
  clocks       - SM clocks and throttle reasons sampled during the run.

`--impl reference` times the float64 oracle instead (there is no other
implementation of this path to run): rank 0 only, a bounded sample of the
same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

_ROOT = os.path.dirname(os.path.abspath(__file__))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

METRIC = "verified draft positions/s at V=128256 bf16; achieved HBM GB/s vs GB300 peak"
UNIT = "positions/s"
V = 128256
TEMPERATURE = 1.0
DATA_SEED = 5          # seed of the synthetic batch on rank 0 (rank r uses DATA_SEED + r)
VERIFY_SEED = 7        # Philox key of the verification uniforms
CSRC = os.path.join(_ROOT, "speculative_decoding_verification_sampling_gb300", "csrc")
TRAFFIC_RECORD = os.path.join(_ROOT, "profiles", "rows_kernels_stoch_b256_k4.md")
# What one call launches at this workload (the library's dispatch): the
# row-parallel kernels, two statistics launches, the residual masses, the sampling.
PATH_KERNELS = "vr_stream (statistics + residual masses) + vr_sample (row-parallel verification, stochastic, bf16)"
REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


# --------------------------------------------------------------------------
# host-side helpers (no GPU needed; covered by CPU tests)
# --------------------------------------------------------------------------
def dist_env() -> tuple[int, int, int]:
    """(rank, world_size, local_rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def replica_seed(rank: int) -> int:
    """Seed of the synthetic batch a rank verifies: replicas hold different sequences."""
    return DATA_SEED + rank


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of `value` over the ranks of the default process group (the value itself alone)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None) -> None:
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and getattr(device, "type", "cpu") == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def needed_rows(accept_len, K: int) -> int:
    """Logit rows the left-to-right rule reads for a batch: a sequence that
    rejects at position j reads target and draft rows 1..j (2j rows); one that
    accepts all K reads K+1 target rows and K draft rows."""
    total = 0
    for L in accept_len:
        L = int(L)
        if L < 0:
            raise ValueError("a sequence reported a data error")
        total += 2 * K + 1 if L >= K else 2 * (L + 1)
    return total


def needed_bytes(accept_len, K: int, V: int, elem_bytes: int) -> int:
    """Algorithmic bytes of one call: the needed logit rows, the drafted
    tokens and the outputs (one read of each, one write of each output)."""
    B = len(accept_len)
    return needed_rows(accept_len, K) * V * elem_bytes + B * K * 4 + B * (K + 1) * 4 + B * 4


def probs_rule_bytes(accept_len, K: int, V: int, elem_bytes: int = 2) -> int:
    """Bytes the left-to-right rule reads with given draft probabilities:
    target rows 0..j (elem_bytes each), p_i(d_i) at every decided position
    (4 bytes), and the float32 probability row only where a draft token is
    rejected (the residual needs it; an accepted position needs p(d) alone)."""
    total = 0
    for L in accept_len:
        L = int(L)
        if L < 0:
            raise ValueError("a sequence reported a data error")
        total += (min(L, K) + 1) * V * elem_bytes + min(L + 1, K) * 4 + (V * 4 if L < K else 0)
    return total


def shortlist_rule_bytes(accept_len, K: int, V: int, lens, one_list: bool, elem_bytes: int = 2) -> int:
    """Bytes the left-to-right rule reads with shortlisted drafts: target rows
    0..j at V, compact draft rows 0..min(j, K-1) at their list lengths
    lens[t], and the int32 lists -- once per sequence when one list serves
    every position (one_list), else each position's list beside its row."""
    total = 0
    for L in accept_len:
        L = int(L)
        if L < 0:
            raise ValueError("a sequence reported a data error")
        npos = min(L + 1, K)
        total += (min(L, K) + 1) * V * elem_bytes + sum(lens[t] for t in range(npos)) * elem_bytes
        total += lens[0] * 4 if one_list else sum(lens[t] for t in range(npos)) * 4
    return total


def kernel_sources_digest() -> str:
    """sha256 over the CUDA and C++ sources of the library, in name order."""
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h", ".cpp")):
            h.update(name.encode())
            with open(os.path.join(CSRC, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()


def recorded_traffic(path: str = TRAFFIC_RECORD, digest: str | None = None):
    """DRAM bytes per verification call from a committed ncu summary, or None
    when the summary is missing or was taken on other kernel sources.  The
    summary holds the lines `traffic_bytes_per_launch: <int>` (per call, all
    its kernels) and `kernel_sources_sha256: <hex>`."""
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_t = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    m_h = re.search(r"kernel_sources_sha256:\s*([0-9a-f]{64})", text)
    if not m_t or not m_h:
        return None
    if m_h.group(1) != (digest or kernel_sources_digest()):
        return None
    return int(m_t.group(1))


def hbm_peak() -> tuple[float, str]:
    """Measured copy bandwidth of this machine's GB300 (GB/s) and where it came from."""
    path = os.path.join(_ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def sm_max_default() -> float | None:
    try:
        with open(os.path.join(_ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["sm_max_mhz"])
    except (OSError, KeyError, ValueError):
        return None


CLOCK_QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_clock_samples(lines) -> list[dict]:
    """Parse `nvidia-smi --format=csv,noheader,nounits` lines of CLOCK_QUERY."""
    out = []
    for line in lines:
        parts = [p.strip() for p in line.strip().split(",")]
        if len(parts) != 9:
            continue
        try:
            sm, smax = float(parts[1]), float(parts[2])
        except ValueError:
            continue
        try:
            util = float(parts[4])
        except ValueError:
            util = float("nan")
        active = [name for name, v in zip(REASONS, parts[5:9]) if v.lower() == "active"]
        out.append({"sm": sm, "sm_max": smax, "util": util, "reasons": active})
    return out


def summarize_clocks(samples: list[dict]) -> dict:
    """Median SM clock over the samples taken under load (all samples when none
    shows load), the maximum clock, and every throttle reason seen."""
    if not samples:
        return {"sm_mhz": None, "sm_max_mhz": sm_max_default(), "reasons": [], "samples": 0,
                "note": "no nvidia-smi sample fell inside the run"}
    loaded = [s for s in samples if not math.isnan(s["util"]) and s["util"] > 0] or samples
    reasons = sorted({r for s in loaded for r in s["reasons"]})
    return {"sm_mhz": statistics.median(s["sm"] for s in loaded),
            "sm_max_mhz": max(s["sm_max"] for s in loaded), "reasons": reasons,
            "samples": len(loaded)}


class ClockSampler:
    """nvidia-smi sampling of this process's GPU every 200 ms while active."""

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.file = None

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={CLOCK_QUERY}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        self.file = tempfile.TemporaryFile(mode="w+")
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
        return False

    def samples(self) -> list[dict]:
        if self.file is None:
            return []
        self.file.seek(0)
        return parse_clock_samples(self.file.readlines())


def workload_name(B: int, K: int) -> str:
    return (f"stochastic verify B={B} K={K} V={V} bf16 T=1; target logits N(0, 2^2), "
            f"draft logits = target + N(0, 0.5^2), drafted tokens sampled from the draft softmax")


def base_line(args, world: int, value: float, ms_per_step: float, B: int, K: int) -> dict:
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name(B, K), "B": B, "K": K, "V": V, "T": TEMPERATURE,
                   "global_batch": B * world, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {args.rotate} device copies of the "
                         f"{(2 * K + 1) * B * V * 2 / 1e6:.0f} MB input set, rotated every step"},
    }


# --------------------------------------------------------------------------
# the float64 oracle on the host cores (reference arm and cpu_baseline)
# --------------------------------------------------------------------------
def oracle_rate(cfg, K: int, seconds: float, n_seq: int | None = None):
    """Positions/s of the oracle over repeated passes on `n_seq` sequences of
    the batch (all of them by default), for at least `seconds` (one pass at least)."""
    import oracle
    B = cfg["draft_tokens"].shape[0]
    n = B if n_seq is None else max(1, min(B, n_seq))
    cores = os.cpu_count() or 1
    tgt, drf, tok = cfg["target"][:n], cfg["draft"][:n], cfg["draft_tokens"][:n]
    passes, t0 = 0, time.perf_counter()
    while True:
        oracle.verify(tgt, drf, tok, TEMPERATURE, VERIFY_SEED, threads=cores)
        passes += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return passes * n * K / el, cores, passes, n, el


def run_reference(args) -> int:
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    import oracle
    from speculative_decoding_verification_sampling_gb300 import synth
    oracle.build()
    B, K = args.batch, args.k
    cfg = synth.throughput(B=B, K=K, seed=replica_seed(0))
    cores = os.cpu_count() or 1
    # size each step so that the whole run stays within about two minutes
    t0 = time.perf_counter()
    probe = min(B, 8)
    oracle.verify(cfg["target"][:probe], cfg["draft"][:probe], cfg["draft_tokens"][:probe], TEMPERATURE,
                  VERIFY_SEED, threads=cores)
    per_seq = (time.perf_counter() - t0) / probe
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(B, budget / max(per_seq, 1e-9))))
    windows = [(s * n) % B for s in range(args.steps + args.warmup)]

    def step(start):
        idx = torch.arange(start, start + n) % B
        oracle.verify(cfg["target"][idx], cfg["draft"][idx], cfg["draft_tokens"][idx], TEMPERATURE,
                      VERIFY_SEED, threads=cores, seq_ids=idx)

    for s in range(args.warmup):
        step(windows[s])
    t0 = time.perf_counter()
    for s in range(args.steps):
        step(windows[args.warmup + s])
    el = time.perf_counter() - t0
    value = n * K * args.steps / el
    line = base_line(args, 1, value, el * 1e3 / args.steps, B, K)
    line["n_gpus"] = world
    line["impl"] = "reference"
    line["dtype"] = "f64"
    sample = (f"{n} of the {B} sequences per step (consecutive windows of the same batch, same "
              f"uniforms), float64 C oracle with {cores} threads")
    line["cpu_baseline"] = {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
    line["e2e"] = {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    line["gpu_launches"] = 0
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# the CUDA path
# --------------------------------------------------------------------------
def run_gb300(args) -> int:
    import torch
    import torch.distributed as dist

    import speculative_decoding_verification_sampling_gb300 as sv
    from speculative_decoding_verification_sampling_gb300 import synth

    rank, world, local_rank = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU path)")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    sv.load()
    B, K = args.batch, args.k

    cfg = synth.throughput(B=B, K=K, seed=replica_seed(rank))
    host_t, host_d, host_k = cfg["target"], cfg["draft"], cfg["draft_tokens"]
    stream = torch.cuda.Stream(dev)
    sets = []
    with torch.cuda.stream(stream):
        t0, d0, k0 = host_t.to(dev), host_d.to(dev), host_k.to(dev)
        sets.append((t0, d0, k0))
        for _ in range(1, args.rotate):
            sets.append((t0.clone(), d0.clone(), k0.clone()))
        outs = [(torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                 torch.empty(B, dtype=torch.int32, device=dev)) for _ in sets]
    stream.synchronize()

    def call(i):
        t, d, k = sets[i % len(sets)]
        ot, ol = outs[i % len(sets)]
        sv.spec_verify(t, d, k, TEMPERATURE, VERIFY_SEED, out_tokens=ot, out_accept_len=ol, stream=stream)

    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    uuid = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else (str(uuid) if uuid else None)

    with ClockSampler(uuid) as clocks:
        with torch.cuda.stream(stream):
            for i in range(max(args.warmup, len(sets))):
                call(i)
        stream.synchronize()
        # every copy of the input set gives the same result
        ref_t, ref_l = outs[0][0].cpu(), outs[0][1].cpu()
        for ot, ol in outs[1:]:
            if not (torch.equal(ot.cpu(), ref_t) and torch.equal(ol.cpu(), ref_l)):
                raise RuntimeError("copies of one input set gave different results")
        alg_bytes = needed_bytes(ref_l.tolist(), K, V, 2)
        all_rows_bytes = (2 * K + 1) * B * V * 2
        mean_len = float(ref_l.double().mean())

        # the K calls run back to back on one stream between one pair of events
        # (an event between two calls would keep the next call's launch from
        # overlapping the end of the one before it)
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        launches0 = sv.spec_launch_count()
        barrier(dev)
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            start.record(stream)
            for i in range(args.steps):
                call(i)
            stop.record(stream)
        torch.cuda.synchronize(dev)
        barrier(dev)
        launches = sv.spec_launch_count() - launches0
        clock_samples = clocks.samples()

    elapsed_ms = start.elapsed_time(stop)
    mean_kernel_s = elapsed_ms / args.steps / 1e3   # this rank's mean duration of one call
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    value = world * B * K * args.steps / (elapsed_ms / 1e3)

    # end to end: pinned host inputs in, results out, every step
    pin_t, pin_d, pin_k = host_t.pin_memory(), host_d.pin_memory(), host_k.pin_memory()
    res_t = torch.empty(B, K + 1, dtype=torch.int32).pin_memory()
    res_l = torch.empty(B, dtype=torch.int32).pin_memory()
    t0, d0, k0 = sets[0]
    ot, ol = outs[0]

    def e2e_step():
        with torch.cuda.stream(stream):
            t0.copy_(pin_t, non_blocking=True)
            d0.copy_(pin_d, non_blocking=True)
            k0.copy_(pin_k, non_blocking=True)
            sv.spec_verify(t0, d0, k0, TEMPERATURE, VERIFY_SEED, out_tokens=ot, out_accept_len=ol, stream=stream)
            res_t.copy_(ot, non_blocking=True)
            res_l.copy_(ol, non_blocking=True)
        stream.synchronize()

    for _ in range(max(3, min(args.warmup, 10))):
        e2e_step()
    e2e_steps = max(3, min(args.steps, 200))
    barrier(dev)
    torch.cuda.synchronize(dev)
    h0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks(time.perf_counter() - h0, dev)
    barrier(dev)
    if not (torch.equal(res_t, ref_t) and torch.equal(res_l, ref_l)):
        raise RuntimeError("end-to-end results differ from the device-resident run")
    h2d = (host_t.numel() * host_t.element_size() + host_d.numel() * host_d.element_size()
           + host_k.numel() * host_k.element_size())
    d2h = res_t.numel() * 4 + res_l.numel() * 4

    if rank == 0:
        line = base_line(args, world, value, elapsed_ms / args.steps, B, K)
        peak, src = hbm_peak()
        achieved = alg_bytes / mean_kernel_s / 1e9
        digest = kernel_sources_digest()
        line["roofline"] = {
            "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": recorded_traffic(digest=digest), "peak_source": src,
            "kernel": PATH_KERNELS, "scope": "the whole verification call (all its kernels), the mean over "
                                             "the timed calls run back to back",
            "algorithmic_bytes_per_launch": alg_bytes, "mean_kernel_us": mean_kernel_s * 1e6,
            "all_rows_bytes_per_launch": all_rows_bytes,
            "all_rows_gbs": all_rows_bytes / mean_kernel_s / 1e9,
        }
        line["e2e"] = {"value": world * B * K * e2e_steps / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "steps": e2e_steps}
        line["gpu_launches"] = int(launches)
        line["clocks"] = summarize_clocks(clock_samples)
        line["emitted_tokens_per_s"] = world * float(ref_l.double().add(1).sum()) * args.steps / (elapsed_ms / 1e3)
        line["mean_accept_len"] = mean_len
        if world == 1 and args.configs:
            del sets, outs
            torch.cuda.empty_cache()
            line["configs"] = config_points(dev, stream)
        if world == 1:
            rate, cores, passes, n, el = oracle_rate(cfg, K, args.cpu_seconds)
            line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                                    "sample": f"{passes} pass(es) of the float64 C oracle over {n} of the "
                                              f"{B} sequences of the same batch, {el:.1f} s"}
        else:
            line["cpu_baseline"] = None
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# --------------------------------------------------------------------------
# every configuration of the benchmark table, timed call by call
# --------------------------------------------------------------------------
def _rule_rows(accept_len, K: int, greedy: bool) -> int:
    """Rows the left-to-right rule reads: stochastic as `needed_rows`; greedy
    reads target rows 0..j (all K + 1 when every draft matches)."""
    if not greedy:
        return needed_rows(accept_len, K)
    return sum(min(int(L), K) + 1 for L in accept_len)


def config_points(dev, stream, calls: int = 40):
    """One record per configuration of the benchmark table (small fp32, greedy,
    Zipf at three draft noises, the shortlisted draft in both layouts, the
    throughput sweep, draft probabilities).  Inputs are made on the device from
    seeded generators; each call is timed alone with CUDA events on the
    launching stream, after a read of 256 MB that evicts the L2 (the smaller
    configurations fit in it).  Bytes: the logits the left-to-right rule reads
    (`rule_bytes`) and every logit row (`all_rows_bytes`)."""
    import torch
    import speculative_decoding_verification_sampling_gb300 as sv
    from speculative_decoding_verification_sampling_gb300 import synth
    peak, src = hbm_peak()
    flush = torch.zeros((2048, 32768), dtype=torch.int32, device=dev)   # 256 MB
    fmax = torch.empty(32768, dtype=torch.int32, device=dev)
    out = []
    errors = []

    def on_copies(call, *tensors):
        """call(*inputs) on device copies of the inputs, enough that a back to
        back run reads at least 300 MB of distinct inputs; None for inputs under
        16 MB (those are timed cold only)."""
        nb = sum(x.numel() * x.element_size() for x in tensors)
        if nb < 16e6:
            return None
        sets = [tuple(x.clone() for x in tensors) for _ in range(max(0, math.ceil(300e6 / nb) - 1))]
        return [lambda x=x: call(*x) for x in sets]

    def timed(fn, more=None):
        """Mean device time of one call: cold (each call alone, after a read of
        256 MB that evicts the L2), and, given calls on copies of the inputs,
        back to back over the copies in turn (the host queued ahead first)."""
        # the inputs were made on the default stream: the calls come after them
        stream.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(stream):
            for _ in range(3):
                r = fn()
            stream.synchronize()
            es = [torch.cuda.Event(enable_timing=True) for _ in range(calls)]
            ee = [torch.cuda.Event(enable_timing=True) for _ in range(calls)]
            for n in range(calls):
                # a read of 256 MB evicts the L2 and leaves no dirty lines behind
                torch.amax(flush, dim=0, out=fmax)
                es[n].record(stream)
                r = fn()
                ee[n].record(stream)
            stream.synchronize()
            cold = statistics.fmean(a.elapsed_time(b) for a, b in zip(es, ee)) * 1e3
            b2b = None
            if more is not None:
                fns = [fn, *more]
                for f in fns:
                    f()
                torch.cuda._sleep(50_000_000)   # a wait on the device while the host queues the calls
                es[0].record(stream)
                for n in range(4 * calls):
                    fns[n % len(fns)]()
                ee[0].record(stream)
                stream.synchronize()
                b2b = es[0].elapsed_time(ee[0]) * 1e3 / (4 * calls)
        return cold, r, b2b

    def record(name, cfg, us, res, elem_bytes, greedy=False, extra_bytes=0, all_rows=None, units=None, b2b=None):
        B, K, V = cfg["B"], cfg["K"], cfg["V"]
        acc = res[1].cpu().tolist()
        bad = [L for L in acc if L < 0]
        if bad:
            # a data error on valid inputs is a fault of the library: report it
            # with the record (the bytes count only the sequences without one)
            errors.append({"workload": name, "sequences": len(bad), "codes": sorted(set(-L for L in bad))})
            acc = [L for L in acc if L >= 0] or [0]
        row_bytes = V * elem_bytes
        rule = _rule_rows(acc, K, greedy) * row_bytes + extra_bytes
        allb = all_rows if all_rows is not None else ((K + 1) if greedy else (2 * K + 1)) * B * row_bytes
        n_units = units if units is not None else B * K
        examined = sum(min(int(L) + 1, K) for L in acc)
        rec = {"workload": name, "B": B, "K": K, "V": V, "us_per_call": us,
               "value": n_units / (us * 1e-6), "unit": "positions/s",
               "mean_accept_len": statistics.fmean(acc), "accept_rate": sum(acc) / max(1, examined),
               "rule_bytes": rule, "all_rows_bytes": allb,
               "roofline": {"bound": "hbm", "achieved": rule / us / 1e3, "peak": peak, "unit": "GB/s",
                            "frac": rule / us / 1e3 / peak, "peak_source": src,
                            "all_rows_gbs": allb / us / 1e3}}
        if b2b is not None:
            rec["back_to_back"] = {"us_per_call": b2b, "value": n_units / (b2b * 1e-6),
                                   "rule_gbs": rule / b2b / 1e3, "frac": rule / b2b / 1e3 / peak}
        out.append(rec)
        return rec

    T1 = TEMPERATURE
    # 1. B=1 K=4 V=32000 fp32
    c = synth.small_stochastic(seed=0, device=dev)
    t, d, k = c["target"], c["draft"], c["draft_tokens"]
    us, r, _ = timed(lambda: sv.spec_verify(t, d, k, 1.0, VERIFY_SEED, stream=stream))
    record("small: B=1 K=4 V=32000 fp32 T=1, target N(0, 2^2), draft = target + N(0, 0.5^2)", c, us, r, 4)
    # 2. greedy B=64 K=5 V=128256 bf16
    c = synth.greedy(device=dev)
    t, k = c["target"], c["draft_tokens"]
    more = on_copies(lambda a, b: sv.spec_verify_greedy(a, b, stream=stream), t, k)
    us, r, b2b = timed(lambda: sv.spec_verify_greedy(t, k, stream=stream), more)
    record("greedy: B=64 K=5 V=128256 bf16 T=0, target N(0, 3^2), drafts = argmax with probability 0.8",
           c, us, r, 2, greedy=True, b2b=b2b)
    del more
    # 3. Zipf B=32 K=7 V=152064 bf16 T=0.7 at three draft noises
    for sigma in (0.25, 0.5, 1.0):
        c = synth.zipf(sigma=sigma, device=dev)
        t, d, k = c["target"], c["draft"], c["draft_tokens"]
        more = on_copies(lambda a, b, e: sv.spec_verify(a, b, e, c["T"], VERIFY_SEED, stream=stream), t, d, k)
        us, r, b2b = timed(lambda: sv.spec_verify(t, d, k, c["T"], VERIFY_SEED, stream=stream), more)
        rec = record(f"zipf: B=32 K=7 V=152064 bf16 T=0.7, draft = target + N(0, {sigma}^2)", c, us, r, 2, b2b=b2b)
        rec["sigma"] = sigma
        del more
    # 4. shortlisted draft, B=64 K=6 V=262144, 32768-token per-sequence lists
    c = synth.shortlist(device=dev)
    Bs, Ks, Vs = c["B"], c["K"], c["V"]
    S = c["shortlist"].shape[1]
    t, d, sl, k = c["target"], c["draft"], c["shortlist"], c["draft_tokens"]
    more = on_copies(lambda a, b, e, f: sv.spec_verify_shortlist(a, b, e, f, 1.0, VERIFY_SEED, stream=stream),
                     t, d, sl, k)
    us, r, b2b = timed(lambda: sv.spec_verify_shortlist(t, d, sl, k, 1.0, VERIFY_SEED, stream=stream), more)
    del more
    acc = r[1].cpu().tolist()
    need = shortlist_rule_bytes(acc, Ks, Vs, [S] * Ks, True)
    rec = record("shortlist (compact): B=64 K=6 V=262144 bf16 T=1, Zipf target, 8 of 64 clusters per sequence "
                 "(S=32768), draft = target + N(0, 0.5^2) on the list", c, us, r, 2,
                 all_rows=Bs * (Ks + 1) * Vs * 2 + Bs * Ks * S * 2 + Bs * S * 4, b2b=b2b)
    rec["rule_bytes"] = need
    rec["roofline"].update(achieved=need / us / 1e3, frac=need / us / 1e3 / peak)
    if b2b is not None:
        rec["back_to_back"].update(rule_gbs=need / b2b / 1e3, frac=need / b2b / 1e3 / peak)
    full = torch.full((Bs, Ks, Vs), float("-inf"), dtype=torch.bfloat16, device=dev)
    full.scatter_(2, sl.long().unsqueeze(1).expand(Bs, Ks, S), d)
    more = on_copies(lambda a, b, e: sv.spec_verify(a, b, e, 1.0, VERIFY_SEED, stream=stream), t, full, k)
    us, r, b2b = timed(lambda: sv.spec_verify(t, full, k, 1.0, VERIFY_SEED, stream=stream), more)
    del more
    record("shortlist (full-vocabulary draft, -inf off the list): B=64 K=6 V=262144 bf16 T=1", c, us, r, 2,
           b2b=b2b)
    del full, t, d, sl, k, c
    # 5. throughput sweep
    for Kp in (4, 8):
        for Bp in (1, 8, 64, 256, 512):
            c = synth.throughput(B=Bp, K=Kp, seed=DATA_SEED, device=dev)
            t, d, k = c["target"], c["draft"], c["draft_tokens"]
            more = on_copies(lambda a, b, e: sv.spec_verify(a, b, e, T1, VERIFY_SEED, stream=stream), t, d, k)
            us, r, b2b = timed(lambda: sv.spec_verify(t, d, k, T1, VERIFY_SEED, stream=stream), more)
            record(f"throughput: B={Bp} K={Kp} V=128256 bf16 T=1", c, us, r, 2, b2b=b2b)
            del t, d, k, c, more
    # draft probabilities at B=256 K=4
    c = synth.throughput(B=256, K=4, seed=DATA_SEED, device=dev)
    t, k = c["target"], c["draft_tokens"]
    probs = torch.softmax(c["draft"].float(), dim=-1)
    del c["draft"]
    more = on_copies(lambda a, b, e: sv.spec_verify(a, b, e, T1, VERIFY_SEED, draft_is_probs=True, stream=stream),
                     t, probs, k)
    us, r, b2b = timed(lambda: sv.spec_verify(t, probs, k, T1, VERIFY_SEED, draft_is_probs=True, stream=stream),
                       more)
    del more
    acc = r[1].cpu().tolist()
    need = probs_rule_bytes(acc, 4, V)
    rec = record("draft probabilities: B=256 K=4 V=128256, bf16 target logits, fp32 draft probabilities", c, us, r,
                 2, all_rows=256 * 5 * V * 2 + 256 * 4 * V * 4, b2b=b2b)
    rec["rule_bytes"] = need
    rec["roofline"].update(achieved=need / us / 1e3, frac=need / us / 1e3 / peak)
    if b2b is not None:
        rec["back_to_back"].update(rule_gbs=need / b2b / 1e3, frac=need / b2b / 1e3 / peak)
    if errors:
        out.append({"data_errors": errors})
    return out


# --------------------------------------------------------------------------
# further workloads of the library (`--workload`), one JSON line each, same keys
# --------------------------------------------------------------------------
def _draft_sample_workload(B: int, K: int, dev):
    """The fused draft-token sampler over the throughput workload's draft rows:
    [B][K][V] bf16 logits, T = 1."""
    import torch
    import oracle.draft_sample as ods
    import speculative_decoding_verification_sampling_gb300 as sv
    from speculative_decoding_verification_sampling_gb300 import synth
    cfg = synth.throughput(B=B, K=K, seed=DATA_SEED)
    host = cfg["draft"]
    nbytes = host.numel() * host.element_size()

    def make_sets(n):
        d0 = host.to(dev)
        return [(d0 if i == 0 else d0.clone(),
                 torch.empty(B, K, dtype=torch.int32, device=dev),
                 torch.empty(B, K, dtype=torch.float32, device=dev)) for i in range(n)]

    def call(st, stream):
        d, ot, op = st
        sv.spec_draft_sample(d, TEMPERATURE, VERIFY_SEED, out_tokens=ot, out_prob=op, stream=stream)

    def result(st):
        return st[1].cpu()

    def oracle_run(i):
        """The oracle on sequence i of the batch: returns the tokens it drew."""
        b = i % B
        ods.draft_sample(host[b:b + 1], TEMPERATURE, VERIFY_SEED, seq_ids=[b])
        return K

    return dict(metric="sampled draft tokens/s at V=128256 bf16 (fused draft-token sampler); achieved HBM GB/s",
                unit="tokens/s", units=B * K, alg_bytes=nbytes + B * K * 8, h2d=nbytes, d2h=B * K * 8,
                make_sets=make_sets, call=call, result=result, host_inputs=[host],
                upload=lambda st: [st[0]], oracle_run=oracle_run,
                kernel="draft_sample_kernel (bf16, T=1)",
                workload=f"draft-token sampling B={B} K={K} V={V} bf16 T=1; draft logits = "
                         f"N(0, 2^2) target + N(0, 0.5^2) (the verification workload's draft rows)",
                l2=f"inputs larger than L2: device copies of the {nbytes / 1e6:.0f} MB draft rows, rotated")


def _kv_commit_workload(B: int, K: int, dev):
    """KV-cache commit after the verification step: a cache shaped like a
    Llama-3-8B one (32 layers, 8 KV heads of 128 dims, keys and values, bf16:
    4096 bytes per entry and layer), capacity 512 entries per sequence, the K
    staged entries of the verification pass, and the accept lengths that the
    verification of the throughput batch returns.  Every step commits at its
    own offsets, so the written entries move through the cache."""
    import numpy as np
    import torch
    import oracle.kv_commit as okv
    import speculative_decoding_verification_sampling_gb300 as sv
    from speculative_decoding_verification_sampling_gb300 import synth
    NL, L, EW = 32, 512, 2048          # EW bf16 elements per entry and layer
    W = EW * 2
    cfg = synth.throughput(B=B, K=K, seed=DATA_SEED)
    _, acc = sv.spec_verify(cfg["target"].to(dev), cfg["draft"].to(dev), cfg["draft_tokens"].to(dev),
                            TEMPERATURE, VERIFY_SEED)
    del cfg
    torch.cuda.synchronize(dev)
    acc_h = acc.cpu()
    committed = int(acc_h.clamp(min=0).sum())
    gen = torch.Generator(device="cpu").manual_seed(DATA_SEED)
    host = torch.randn((NL, B, K, EW), generator=gen).to(torch.bfloat16)
    cache = torch.zeros((NL, B, L, EW), dtype=torch.bfloat16, device=dev)
    # one length array per call (the commit advances it in place): step i
    # commits sequence b at entry (7 b + 11 i) mod (L - K)
    n_calls = 4096
    steps = torch.arange(n_calls)[:, None]
    lens = ((torch.arange(B)[None, :] * 7 + 11 * steps) % (L - K)).to(torch.int32).to(dev)
    state = {"step": 0}

    def make_sets(n):
        s0 = host.to(dev)
        return [s0 if i == 0 else s0.clone() for i in range(n)]

    def call(st, stream):
        i = state["step"] % n_calls
        state["step"] += 1
        sv.spec_kv_commit(cache, st, acc, lens[i], stream=stream)

    def result(st):
        return torch.zeros(1)

    cache_h = np.zeros((NL, 1, L, W), dtype=np.uint8)
    staged_h = host.view(torch.uint8).numpy()

    def oracle_run(i):
        b = i % B
        okv.kv_commit(cache_h, staged_h[:, b:b + 1], [0], [int(acc_h[b])])
        return max(0, int(acc_h[b])) * NL

    return dict(metric="committed KV entries/s (entries x layers; 4096-byte bf16 entries, 32 layers, "
                       "accept lengths of the B=256 K=4 verification); achieved HBM GB/s",
                unit="entries/s", units=committed * NL, alg_bytes=2 * committed * NL * W + 2 * B * 4,
                h2d=host.numel() * 2, d2h=4 * B, make_sets=make_sets, call=call, result=result,
                host_inputs=[host], upload=lambda st: [st], oracle_run=oracle_run,
                kernel="kv_copy + kv_len",
                workload=f"KV-cache commit B={B} K={K}: cache [32][{B}][{L}][4096 B] bf16, staged "
                         f"[32][{B}][{K}][4096 B], accept lengths of the verification step "
                         f"(mean {float(acc_h.double().mean()):.2f})",
                l2="staged entries rotated over device copies; each step commits at new offsets")


def _tree_greedy_workload(B: int, K: int, dev):
    """Greedy verification of an EAGLE-style draft tree: 32 sequences, top-k
    branches (4, 2, 2, 1, 1) per depth (61 nodes), V=128256 bf16 target rows
    ~ N(0, 3^2); every node row is read (500 MB per call).  K is not used."""
    import torch
    import oracle.tree as otr
    import speculative_decoding_verification_sampling_gb300 as sv
    from speculative_decoding_verification_sampling_gb300 import synth
    Bt = 32
    cfg = synth.tree_greedy(B=Bt, V=V, seed=DATA_SEED)
    host_t, host_k, host_p = cfg["target"], cfg["tree_tokens"], cfg["parent"]
    N = cfg["N"]
    nbytes = host_t.numel() * host_t.element_size()
    ws = torch.empty(sv.load().spec_tree_workspace_bytes(Bt, N, V), dtype=torch.uint8, device=dev)

    def make_sets(n):
        t0, k0, p0 = host_t.to(dev), host_k.to(dev), host_p.to(dev)
        return [((t0, k0, p0) if i == 0 else (t0.clone(), k0.clone(), p0.clone())) + ([None],) for i in range(n)]

    def call(st, stream):
        t, k, p, out = st
        out[0] = sv.spec_verify_tree_greedy(t, k, p, workspace=ws, stream=stream)

    def result(st):
        return st[3][0][2].cpu()

    def oracle_run(i):
        b = i % Bt
        otr.tree_verify_greedy(host_t[b:b + 1], host_k[b:b + 1].numpy(), host_p[b:b + 1].numpy())
        return N - 1

    return dict(metric="verified draft-tree nodes/s (greedy tree verification, 61-node trees, V=128256 bf16); "
                       "achieved HBM GB/s", unit="nodes/s", units=Bt * (N - 1),
                alg_bytes=nbytes + Bt * N * 8 + Bt * N * 8 + Bt * 4, h2d=nbytes + Bt * N * 8, d2h=Bt * (2 * N + 1) * 4,
                make_sets=make_sets, call=call, result=result, host_inputs=[host_t, host_k, host_p],
                upload=lambda st: [st[0], st[1], st[2]], oracle_run=oracle_run,
                kernel="draft_sample_kernel (greedy, node rows) + tree_walk", B=Bt, K=N - 1,
                workload=f"greedy tree verification B={Bt} N={N} (branching 4,2,2,1,1) V={V} bf16; target "
                         f"N(0, 3^2); first children hold the argmax with probability 0.7",
                l2=f"inputs larger than L2: device copies of the {nbytes / 1e6:.0f} MB node rows, rotated")


def _shortlist_pos_workload(B: int, K: int, dev):
    """Verification with per-position shortlists: B=64, K=6, V=262144 bf16,
    Zipf target, 64 clusters of 4096 tokens, the DynaSpec position-aware budget
    with k_max = 8 (8, 8, 1, 1, 1, 1 clusters per draft step), draft = target +
    N(0, 0.5^2) on each list (compact rows of up to 32768 logits)."""
    import torch
    import oracle
    import speculative_decoding_verification_sampling_gb300 as sv
    from speculative_decoding_verification_sampling_gb300 import synth
    Bs, Ks, Vs = 64, 6, 262144
    cfg = synth.shortlist_per_position(B=Bs, K=Ks, V=Vs, seed=DATA_SEED)
    lens = cfg["shortlist_len"]
    S = cfg["S"]
    host = [cfg["target"], cfg["draft"], cfg["shortlist"], cfg["draft_tokens"]]
    nbytes = sum(h.numel() * h.element_size() for h in host)
    ref = oracle.verify(cfg["target"], cfg["draft"], cfg["draft_tokens"], TEMPERATURE, VERIFY_SEED,
                        shortlist=cfg["shortlist"], shortlist_len=lens)
    # bytes the left-to-right rule reads: target rows 0..j, draft rows and lists 0..min(j, K-1)
    need = shortlist_rule_bytes(ref["accept_len"].tolist(), Ks, Vs, lens, False)
    need += Bs * (Ks * 4 + (Ks + 1) * 4 + 4)

    def make_sets(n):
        d0 = [h.to(dev) for h in host]
        return [(d0 if i == 0 else [x.clone() for x in d0]) + [None] for i in range(n)]

    def call(st, stream):
        t, d, sl, k, _ = st
        st[4] = sv.spec_verify_shortlist_pos(t, d, sl, k, TEMPERATURE, VERIFY_SEED, shortlist_len=lens,
                                             stream=stream)

    def result(st):
        return st[4][0].cpu()

    def oracle_run(i):
        b = i % Bs
        oracle.verify(cfg["target"][b:b + 1], cfg["draft"][b:b + 1], cfg["draft_tokens"][b:b + 1], TEMPERATURE,
                      VERIFY_SEED, shortlist=cfg["shortlist"][b:b + 1], shortlist_len=lens, seq_ids=[b],
                      threads=1)
        return Ks

    return dict(metric="verified draft positions/s with per-position shortlists (DynaSpec budget, V=262144 "
                       "bf16); achieved HBM GB/s", unit="positions/s", units=Bs * Ks, alg_bytes=need,
                h2d=nbytes, d2h=Bs * (Ks + 2) * 4, make_sets=make_sets, call=call, result=result,
                host_inputs=host, upload=lambda st: st[:4], oracle_run=oracle_run,
                kernel="vr_stats x2 + vr_residual + vr_sample (row-parallel, per-position shortlists)",
                B=Bs, K=Ks,
                workload=f"per-position shortlists B={Bs} K={Ks} V={Vs} bf16 T=1: Zipf target, 64 clusters "
                         f"of 4096, budget (8, 8, 1, 1, 1, 1) clusters, list lengths {lens}, draft = "
                         f"target + N(0, 0.5^2) on the lists",
                l2=f"inputs larger than L2: device copies of the {nbytes / 1e6:.0f} MB input set, rotated")


def _greedy_workload(B: int, K: int, dev):
    """Greedy verification (the benchmark table's config 2): B=64, K=5,
    V=128256 bf16, target ~ N(0, 3^2), drafted tokens = the argmax with
    probability 0.8.  B and K are fixed by the configuration."""
    import torch
    import oracle
    import speculative_decoding_verification_sampling_gb300 as sv
    from speculative_decoding_verification_sampling_gb300 import synth
    Bg, Kg = 64, 5
    cfg = synth.greedy(B=Bg, K=Kg, V=V, seed=DATA_SEED)
    host_t, host_k = cfg["target"], cfg["draft_tokens"]
    nbytes = host_t.numel() * host_t.element_size()
    ref = oracle.verify(host_t, None, host_k, 0.0, 0)
    need = _rule_rows(ref["accept_len"].tolist(), Kg, True) * V * 2 + Bg * Kg * 4 + Bg * (Kg + 2) * 4
    ws = torch.zeros(sv.spec_workspace_bytes(Bg, Kg, V), dtype=torch.uint8, device=dev)

    def make_sets(n):
        t0, k0 = host_t.to(dev), host_k.to(dev)
        return [[t0 if i == 0 else t0.clone(), k0, torch.empty(Bg, Kg + 1, dtype=torch.int32, device=dev),
                 torch.empty(Bg, dtype=torch.int32, device=dev)] for i in range(max(n, 4))]

    def call(st, stream):
        t, k, ot, ol = st
        sv.spec_verify_greedy(t, k, out_tokens=ot, out_accept_len=ol, workspace=ws, stream=stream)

    def result(st):
        return torch.cat([st[2].flatten(), st[3]]).cpu()

    def oracle_run(i):
        b = i % Bg
        oracle.verify(host_t[b:b + 1], None, host_k[b:b + 1], 0.0, 0)
        return Kg

    return dict(metric="verified draft positions/s (greedy, V=128256 bf16); achieved HBM GB/s", unit="positions/s",
                units=Bg * Kg, alg_bytes=need, h2d=nbytes + Bg * Kg * 4, d2h=Bg * (Kg + 2) * 4, make_sets=make_sets,
                call=call, result=result, host_inputs=[host_t, host_k], upload=lambda st: st[:2],
                oracle_run=oracle_run, kernel="vg_bulk (one launch: argmax of every target row, the walk)",
                B=Bg, K=Kg,
                workload=f"greedy B={Bg} K={Kg} V={V} bf16 T=0: target N(0, 3^2), drafts = argmax with "
                         f"probability 0.8",
                l2=f"inputs larger than L2: device copies of the {nbytes / 1e6:.0f} MB target rows, rotated")


def _small_workload(B: int, K: int, dev):
    """The smallest call of the benchmark table (config 1): B=1, K=4,
    V=32000 float32, T=1, target ~ N(0, 2^2), draft = target + N(0, 0.5^2):
    a latency figure.  Enough device copies of the 1.15 MB input set are
    rotated that the calls read more than twice the L2."""
    import torch
    import oracle
    import speculative_decoding_verification_sampling_gb300 as sv
    from speculative_decoding_verification_sampling_gb300 import synth
    cfg = synth.small_stochastic(seed=DATA_SEED)
    Bs, Ks, Vs = 1, 4, 32000
    host = [cfg["target"], cfg["draft"], cfg["draft_tokens"]]
    nbytes = sum(h.numel() * h.element_size() for h in host)
    ref = oracle.verify(cfg["target"], cfg["draft"], cfg["draft_tokens"], TEMPERATURE, VERIFY_SEED)
    need = needed_bytes(ref["accept_len"].tolist(), Ks, Vs, 4)
    ws = torch.zeros(sv.spec_workspace_bytes(Bs, Ks, Vs), dtype=torch.uint8, device=dev)
    copies = math.ceil(2 * 129e6 / nbytes)

    def make_sets(n):
        d0 = [h.to(dev) for h in host]
        return [(d0 if i == 0 else [x.clone() for x in d0]) +
                [torch.empty(Bs, Ks + 1, dtype=torch.int32, device=dev), torch.empty(Bs, dtype=torch.int32, device=dev)]
                for i in range(max(n, copies))]

    def call(st, stream):
        t, d, k, ot, ol = st
        sv.spec_verify(t, d, k, TEMPERATURE, VERIFY_SEED, out_tokens=ot, out_accept_len=ol, workspace=ws,
                       stream=stream)

    def result(st):
        return torch.cat([st[3].flatten(), st[4]]).cpu()

    def oracle_run(i):
        oracle.verify(cfg["target"], cfg["draft"], cfg["draft_tokens"], TEMPERATURE, VERIFY_SEED)
        return Ks

    return dict(metric="verified draft positions/s (B=1 K=4 V=32000 fp32: latency per call); achieved HBM GB/s",
                unit="positions/s", units=Bs * Ks, alg_bytes=need, h2d=nbytes, d2h=Bs * (Ks + 2) * 4,
                make_sets=make_sets, call=call, result=result, host_inputs=host, upload=lambda st: st[:3],
                oracle_run=oracle_run, kernel="vr_resident + vr_sample (every row held in shared memory)",
                B=Bs, K=Ks, V=Vs, dtype="f32",
                workload=f"small B={Bs} K={Ks} V={Vs} fp32 T=1: target N(0, 2^2), draft = target + N(0, 0.5^2)",
                l2=f"inputs larger than L2 in turn: {copies} device copies of the {nbytes / 1e6:.2f} MB input set, "
                   f"rotated")


def _shortlist_workload(B: int, K: int, dev):
    """The shortlisted configuration of the benchmark table (config 4): B=64,
    K=6, V=262144 bf16, Zipf target, 8 of 64 clusters of 4096 tokens per
    sequence (S=32768, compact draft rows), draft = target + N(0, 0.5^2) on
    the list.  B and K are fixed by the configuration."""
    import torch
    import oracle
    import speculative_decoding_verification_sampling_gb300 as sv
    from speculative_decoding_verification_sampling_gb300 import synth
    cfg = synth.shortlist(seed=DATA_SEED)
    Bs, Ks, Vs = cfg["B"], cfg["K"], cfg["V"]
    S = cfg["shortlist"].shape[1]
    host = [cfg["target"], cfg["draft"], cfg["shortlist"], cfg["draft_tokens"]]
    nbytes = sum(h.numel() * h.element_size() for h in host)
    ref = oracle.verify(cfg["target"], cfg["draft"], cfg["draft_tokens"], TEMPERATURE, VERIFY_SEED,
                        shortlist=cfg["shortlist"])
    need = shortlist_rule_bytes(ref["accept_len"].tolist(), Ks, Vs, [S] * Ks, True)
    ws = torch.zeros(sv.spec_workspace_bytes(Bs, Ks, Vs, S), dtype=torch.uint8, device=dev)

    def make_sets(n):
        d0 = [h.to(dev) for h in host]
        return [(d0 if i == 0 else [x.clone() for x in d0]) + [None] for i in range(max(n, 2))]

    def call(st, stream):
        t, d, sl, k, _ = st
        st[4] = sv.spec_verify_shortlist(t, d, sl, k, TEMPERATURE, VERIFY_SEED, workspace=ws, stream=stream)

    def result(st):
        return st[4][1].cpu()

    def oracle_run(i):
        b = i % Bs
        oracle.verify(cfg["target"][b:b + 1], cfg["draft"][b:b + 1], cfg["draft_tokens"][b:b + 1], TEMPERATURE,
                      VERIFY_SEED, shortlist=cfg["shortlist"][b:b + 1], seq_ids=[b], threads=1)
        return Ks

    return dict(metric="verified draft positions/s with a per-sequence shortlisted draft (V=262144 bf16); "
                       "achieved HBM GB/s", unit="positions/s", units=Bs * Ks, alg_bytes=need, h2d=nbytes,
                d2h=Bs * (Ks + 2) * 4, make_sets=make_sets, call=call, result=result, host_inputs=host,
                upload=lambda st: st[:4], oracle_run=oracle_run,
                kernel="vr_stats x2 + vr_residual + vr_sample (row-parallel, shortlisted draft)", B=Bs, K=Ks, V=Vs,
                workload=f"shortlist B={Bs} K={Ks} V={Vs} S={S} bf16 T=1: Zipf target, 8 of 64 clusters of 4096 "
                         f"per sequence, draft = target + N(0, 0.5^2) on the list",
                l2=f"inputs larger than L2: device copies of the {nbytes / 1e6:.0f} MB input set, rotated")


def _probs_workload(B: int, K: int, dev):
    """Draft probabilities: B=256, K=4, V=128256, bf16 target logits and
    float32 draft probabilities (the softmax of the throughput workload's
    draft logits), T=1.  B and K are fixed."""
    import torch
    import oracle
    import speculative_decoding_verification_sampling_gb300 as sv
    from speculative_decoding_verification_sampling_gb300 import synth
    Bp, Kp = 256, 4
    cfg = synth.throughput(B=Bp, K=Kp, seed=DATA_SEED)
    probs = torch.softmax(cfg["draft"].float(), dim=-1)
    host = [cfg["target"], probs, cfg["draft_tokens"]]
    nbytes = sum(h.numel() * h.element_size() for h in host)
    ref = oracle.verify(cfg["target"], probs, cfg["draft_tokens"], TEMPERATURE, VERIFY_SEED, draft_is_probs=True)
    need = probs_rule_bytes(ref["accept_len"].tolist(), Kp, V)
    ws = torch.zeros(sv.spec_workspace_bytes(Bp, Kp, V), dtype=torch.uint8, device=dev)

    def make_sets(n):
        d0 = [h.to(dev) for h in host]
        return [(d0 if i == 0 else [x.clone() for x in d0]) + [None] for i in range(max(n, 2))]

    def call(st, stream):
        t, d, k, _ = st
        st[3] = sv.spec_verify(t, d, k, TEMPERATURE, VERIFY_SEED, draft_is_probs=True, workspace=ws, stream=stream)

    def result(st):
        return st[3][1].cpu()

    def oracle_run(i):
        b = i % Bp
        oracle.verify(cfg["target"][b:b + 1], probs[b:b + 1], cfg["draft_tokens"][b:b + 1], TEMPERATURE,
                      VERIFY_SEED, draft_is_probs=True, seq_ids=[b], threads=1)
        return Kp

    return dict(metric="verified draft positions/s with draft probabilities (V=128256, bf16 target, fp32 "
                       "probabilities); achieved HBM GB/s", unit="positions/s", units=Bp * Kp, alg_bytes=need,
                h2d=nbytes, d2h=Bp * (Kp + 2) * 4, make_sets=make_sets, call=call, result=result, host_inputs=host,
                upload=lambda st: st[:3], oracle_run=oracle_run,
                kernel="vr_stream<BF16, probabilities> + vr_sample (target rows streamed, p(d) at the decision)",
                B=Bp, K=Kp,
                workload=f"draft probabilities B={Bp} K={Kp} V={V}: bf16 target N(0, 2^2), fp32 probabilities of "
                         f"target + N(0, 0.5^2), T=1",
                l2=f"inputs larger than L2: device copies of the {nbytes / 1e6:.0f} MB input set, rotated")


EXTRA_WORKLOADS = {"shortlist_pos": _shortlist_pos_workload,
                   "draft_sample": _draft_sample_workload, "kv_commit": _kv_commit_workload,
                   "tree_greedy": _tree_greedy_workload, "greedy": _greedy_workload, "small": _small_workload,
                   "shortlist": _shortlist_workload, "probs": _probs_workload}


def run_extra(args) -> int:
    """A further workload of the library, timed like the verification step."""
    import torch
    import torch.distributed as dist
    import speculative_decoding_verification_sampling_gb300 as sv

    rank, world, local_rank = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU path)")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    sv.load()
    w = EXTRA_WORKLOADS[args.workload](args.batch, args.k, dev)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        sets = w["make_sets"](args.rotate)
    stream.synchronize()
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    uuid = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else (str(uuid) if uuid else None)
    with ClockSampler(uuid) as clocks:
        with torch.cuda.stream(stream):
            for i in range(max(args.warmup, len(sets))):
                w["call"](sets[i % len(sets)], stream)
        stream.synchronize()
        ref = w["result"](sets[0])
        for st in sets[1:]:
            if not torch.equal(w["result"](st), ref):
                raise RuntimeError("copies of one input set gave different results")
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        launches0 = sv.spec_launch_count()
        barrier(dev)
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            start.record(stream)
            for i in range(args.steps):
                w["call"](sets[i % len(sets)], stream)
            stop.record(stream)
        torch.cuda.synchronize(dev)
        barrier(dev)
        launches = sv.spec_launch_count() - launches0
        clock_samples = clocks.samples()
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), dev)
    mean_s = elapsed_ms / args.steps / 1e3
    value = world * w["units"] * args.steps / (elapsed_ms / 1e3)

    # end to end: inputs copied in from pinned host memory, results read back, every step
    pinned = [h.pin_memory() for h in w["host_inputs"]]
    st0 = sets[0]

    def e2e_step():
        with torch.cuda.stream(stream):
            for dst, src in zip(w["upload"](st0), pinned):
                dst.copy_(src, non_blocking=True)
            w["call"](st0, stream)
            out = w["result"](st0)
        stream.synchronize()
        return out

    for _ in range(3):
        e2e_step()
    e2e_steps = max(3, min(args.steps, 100))
    barrier(dev)
    h0 = time.perf_counter()
    for _ in range(e2e_steps):
        last = e2e_step()
    e2e_s = max_over_ranks(time.perf_counter() - h0, dev)
    if not torch.equal(last, ref):
        raise RuntimeError("end-to-end results differ from the device-resident run")
    if rank == 0:
        peak, src = hbm_peak()
        achieved = w["alg_bytes"] / mean_s / 1e9
        line = {
            "metric": w["metric"], "value": value, "unit": w["unit"], "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.get("dtype", "bf16"), "data": "synthetic",
            "config": {"workload": w["workload"], "B": w.get("B", args.batch), "K": w.get("K", args.k),
                       "V": w.get("V", V),
                       "parallelism": f"replicas x{world}", "l2": w["l2"]},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": None, "peak_source": src, "kernel": w["kernel"],
                         "algorithmic_bytes_per_launch": w["alg_bytes"], "mean_kernel_us": mean_s * 1e6},
            "e2e": {"value": world * w["units"] * e2e_steps / e2e_s, "unit": w["unit"],
                    "h2d_bytes_per_step": w["h2d"], "d2h_bytes_per_step": w["d2h"], "steps": e2e_steps},
            "gpu_launches": int(launches),
            "clocks": summarize_clocks(clock_samples),
        }
        if world == 1 and args.cpu_seconds > 0:
            t0, n, i = time.perf_counter(), 0, 0
            while time.perf_counter() - t0 < args.cpu_seconds:
                n += w["oracle_run"](i)
                i += 1
            el = time.perf_counter() - t0
            line["cpu_baseline"] = {"value": n / el, "unit": w["unit"], "cores": 1, "kind": "oracle",
                                    "sample": f"{n} units of the same workload through the float64 oracle "
                                              f"(one thread), {el:.1f} s"}
        else:
            line["cpu_baseline"] = None
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--batch", type=int, default=256, help="sequences per GPU")
    ap.add_argument("--k", type=int, default=4, help="drafted tokens per sequence")
    ap.add_argument("--rotate", type=int, default=4, help="device copies of the input set")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="length of the oracle sample")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="leave out the per-configuration records (one GPU only)")
    ap.add_argument("--workload", choices=("verify",) + tuple(EXTRA_WORKLOADS), default="verify",
                    help="the verification step (default), or a further workload of the library")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    _, world, _ = dist_env()
    if world != args.gpus:
        if world == 1 and args.gpus > 1:
            ap.error("--gpus N > 1 runs under torchrun with N processes")
    if args.impl == "reference":
        return run_reference(args)
    if args.workload != "verify":
        return run_extra(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
