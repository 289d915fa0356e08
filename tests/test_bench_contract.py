"""bench.py's output contract, checked on CPU through its reference arm (the
fp64 oracle timed on the host): one JSON line with the keys the benchmark
contract names, the same metric and unit as the GPU arm for the same
workload, and an e2e entry that copies nothing."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
        "cpu_baseline", "e2e"}


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,metric,unit", [
    ("b1_h2_n128_d64", bench.METRIC, "TFLOP/s"),
    ("decode_b32_h32_nq1_nk8192_d128", bench.DECODE_METRIC, "GB/s"),
])
def test_reference_arm_line(workload, metric, unit):
    d = _run("--impl", "reference", "--workload", workload, "--steps", "1", "--warmup", "3")
    assert KEYS <= set(d), sorted(KEYS - set(d))
    assert d["impl"] == "reference"
    assert d["metric"] == metric and d["unit"] == unit
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"].startswith(workload)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == unit
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_workload_tables_are_consistent():
    """Every named workload has positive sizes; the GPT-style sweeps keep
    B * N = 16384 tokens; no name appears in two tables."""
    names = set(bench.WORKLOADS)
    assert not names & set(bench.VARLEN_WORKLOADS)
    assert not names & set(bench.DECODE_WORKLOADS)
    assert bench.DEFAULT_WORKLOAD in bench.WORKLOADS
    for name, (B, H, N, d) in bench.WORKLOADS.items():
        assert min(B, H, N) >= 1 and d in (32, 64, 96, 128, 256), name
        if name.startswith("gpt_"):
            assert B * N == 16384, name
    for name, (B, H, Nq, Nk, d) in bench.DECODE_WORKLOADS.items():
        assert 1 <= Nq <= 16 and Nk >= 1 and d in (32, 64, 96, 128), name
