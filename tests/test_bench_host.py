"""Host-side logic of bench.py (no GPU): aggregation over ranks with a real
2-process gloo group, clock-record parsing, the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_aggregate_counts_every_rank_over_the_slowest_time():
    # 2 ranks x 10 steps x 1e12 FLOP in 4 s (slowest rank) = 5 TFLOP/s
    assert bench.aggregate(10**12, 10, 4.0, 2) == pytest.approx(5.0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import bench
world, rank, local = bench.dist_setup(2)
bench.barrier(world)
t = bench.max_over_ranks(1.0 + rank * 2.5, world)
v = bench.aggregate(10**12, 4, t, world)
print(json.dumps({{"rank": rank, "max": t, "value": v}}))
import torch.distributed as dist
dist.destroy_process_group()
"""


def test_max_over_ranks_with_two_gloo_ranks():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (out, err) in zip(procs, outs):
        assert p.returncode == 0, err
    res = [json.loads(o.strip().splitlines()[-1]) for o, _ in outs]
    for r in res:
        assert r["max"] == pytest.approx(3.5)            # slowest rank's time
        assert r["value"] == pytest.approx(2 * 4 / 3.5)  # both ranks' work


def test_clock_summary_parses_nvidia_smi_lines():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.lines = [
        "2026/12/02 10:00:00.000, 1965, 2070, 900.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:00:00.100, 1440, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:00:00.200, 1500, 2070, 1380.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage",
    ]
    d = s.summary()
    assert d["samples"] == 3 and d["sm_mhz"] == 1500 and d["sm_max_mhz"] == 2070
    assert d["reasons"] == ["sw_power_cap"]


def test_reference_arm_prints_the_contract_fields():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3", "--workload", "qwen2.5-0.5b-mlp-m128"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in line
    assert line["impl"] == "reference" and line["steps"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["config"]["workload"] == "qwen2.5-0.5b-mlp-m128"


def test_reference_arm_non_zero_rank_does_nothing():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2"], capture_output=True, text=True, timeout=120, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_profiled_traffic_reads_both_record_forms(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    stamp = bench.source_stamp()
    (prof / "one.md").write_text(
        "text\nbench-key kernel=k_a\nbench-key workload=w1\n"
        f"bench-key source_stamp={stamp}\nbench-key dram_bytes_per_launch=100\n")
    (prof / "many.md").write_text(
        f"bench-key kernel=k_b<fp8> workload=w1 source_stamp={stamp} dram_bytes_per_launch=200\n"
        f"bench-key kernel=k_b<fp8> workload=w2 source_stamp=0000 dram_bytes_per_launch=300\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_stamp", lambda: stamp)
    assert bench.profiled_traffic("k_a", "w1")[0] == 100.0
    assert bench.profiled_traffic("k_b<fp8>", "w1")[0] == 200.0
    assert bench.profiled_traffic("k_b<fp8>", "w2") == (None, None)  # stale stamp
    assert bench.profiled_traffic("k_a", "w2") == (None, None)


def test_source_stamp_ignores_comments_not_code(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", ["k.cu"])
    src.write_text("int f(int x) {  // doubles x\n  return 2 * x;\n}\n")
    base = bench.source_stamp()
    src.write_text("/* a block\n   comment */\nint f(int x) {  // twice x\n\n  return 2 * x;\n}\n")
    assert bench.source_stamp() == base  # comments and blank lines only
    src.write_text("int f(int x) {  // doubles x\n  return 3 * x;\n}\n")
    assert bench.source_stamp() != base  # a code change
    assert bench._code_only("a = 1;  // c\n/* x */ b = 2;\n") == "a = 1;\n b = 2;"
