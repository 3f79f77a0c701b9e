"""Host-side logic of bench.py: byte accounting, clock parsing, the traffic
record, and the multi-process paths (gloo ranks on the CPU)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_needed_rows_follow_the_left_to_right_rule():
    K = 4
    # rejection at the first draft: target row 1 and draft row 1
    assert bench.needed_rows([0], K) == 2
    # two accepted, rejection at the third: rows 1..3 of each
    assert bench.needed_rows([2], K) == 6
    # every draft accepted: K+1 target rows, K draft rows
    assert bench.needed_rows([4], K) == 9
    assert bench.needed_rows([0, 2, 4, 3], K) == 2 + 6 + 9 + 8
    with pytest.raises(ValueError):
        bench.needed_rows([-2], K)


def test_needed_bytes_counts_rows_tokens_and_outputs():
    B, K, V = 3, 2, 10
    got = bench.needed_bytes([0, 1, 2], K, V, 2)
    rows = 2 + 4 + 5
    assert got == rows * V * 2 + B * K * 4 + B * (K + 1) * 4 + B * 4


def test_probability_rule_bytes_read_the_row_only_at_a_rejection():
    K, V = 2, 10
    # rejection at the first draft: target row 0 (20 B), p(d) once, the probability row (40 B)
    assert bench.probs_rule_bytes([0], K, V) == 20 + 4 + 40
    # rejection at the second: target rows 0..1, p(d) twice, the probability row
    assert bench.probs_rule_bytes([1], K, V) == 40 + 8 + 40
    # every draft accepted: K + 1 target rows and p(d) at each position, no probability row
    assert bench.probs_rule_bytes([2], K, V) == 60 + 8
    assert bench.probs_rule_bytes([0, 1, 2], K, V) == 64 + 88 + 68
    with pytest.raises(ValueError):
        bench.probs_rule_bytes([-2], K, V)


def test_shortlist_rule_bytes_count_rows_at_their_list_lengths():
    K, V = 2, 10
    # one list per sequence (4 entries): read once, 16 B
    assert bench.shortlist_rule_bytes([0], K, V, [4, 4], True) == 20 + 8 + 16
    assert bench.shortlist_rule_bytes([2], K, V, [4, 4], True) == 60 + 16 + 16
    # a list per position (4 and 2 entries), each read with its row
    assert bench.shortlist_rule_bytes([1], K, V, [4, 2], False) == 40 + 12 + 24
    assert bench.shortlist_rule_bytes([0], K, V, [4, 2], False) == 20 + 8 + 16
    with pytest.raises(ValueError):
        bench.shortlist_rule_bytes([-1], K, V, [4, 4], True)


def test_clock_samples_parse_and_summarize():
    lines = [
        "2026/12/02 10:00:00.000, 1965, 2070, 900.1, 100, Not Active, Not Active, Not Active, Active\n",
        "2026/12/02 10:00:00.200, 1980, 2070, 910.0, 99, Not Active, Not Active, Not Active, Not Active\n",
        "2026/12/02 10:00:00.400, 345, 2070, 120.0, 0, Not Active, Not Active, Not Active, Not Active\n",
        "garbage line\n",
    ]
    s = bench.parse_clock_samples(lines)
    assert len(s) == 3
    c = bench.summarize_clocks(s)
    assert c["sm_mhz"] == pytest.approx((1965 + 1980) / 2)   # idle sample left out
    assert c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]
    assert bench.summarize_clocks([])["samples"] == 0


def test_traffic_record_needs_matching_sources(tmp_path):
    digest = bench.kernel_sources_digest()
    p = tmp_path / "rec.md"
    p.write_text(f"traffic_bytes_per_launch: 123456\nkernel_sources_sha256: {digest}\n")
    assert bench.recorded_traffic(str(p)) == 123456
    p.write_text(f"traffic_bytes_per_launch: 123456\nkernel_sources_sha256: {'0' * 64}\n")
    assert bench.recorded_traffic(str(p)) is None
    assert bench.recorded_traffic(str(tmp_path / "missing.md")) is None


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    bench.barrier()
    m = bench.max_over_ranks(10.0 + 5.0 * rank)
    q.put((r, w, lr, m, bench.replica_seed(r)))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world_size_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1]
    assert all(x[1] == 2 for x in res)
    assert all(x[3] == 15.0 for x in res)          # the slowest rank decides
    assert res[0][4] != res[1][4]                  # replicas verify different batches


def test_single_process_max_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3", "--batch", "2", "--k", "2"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["metric"] == bench.METRIC and rec["unit"] == "positions/s"
    assert rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["d2h_bytes_per_step"] == 0
    assert rec["n_gpus"] == 2 and rec["steps"] == 2
