"""bench.py's GPU arm on small workloads: one JSON line carrying every key of
the benchmark contract, with a roofline entry whose fraction follows from its
own figures, an end-to-end entry that copies the step's inputs and outputs,
the count of this library's launches, the sampled clocks and the CUDA-graph
replay of the same step."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

pytestmark = pytest.mark.gpu

KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
        "e2e", "gpu_launches", "clocks", "graph"}


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args,
                        "--no-cpu-baseline", "--no-extra-legs", "--e2e-steps", "2"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def _common(d, steps, launches_per_step):
    assert KEYS <= set(d), sorted(KEYS - set(d))
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["steps"] == steps and d["warmup"] == 3 and d["dtype"] == "bf16"
    assert d["gpu_launches"] == launches_per_step * steps
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) <= 1e-9 * max(1.0, r["frac"])
    e = d["e2e"]
    assert e["unit"] == d["unit"] and e["value"] > 0
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["clocks"]["sm_max_mhz"] is None or d["clocks"]["sm_max_mhz"] > 0
    assert d["graph"]["ms_per_step"] > 0 and d["graph"]["fwd_bwd_tflops"] > 0


@pytest.mark.parametrize("causal", [False, True])
def test_dense_line(causal):
    args = ["--workload", "b4_h8_n1024_d64", "--steps", "4", "--warmup", "3"]
    d = _run(*args, *(["--causal"] if causal else []))
    _common(d, 4, 4)
    assert d["config"]["workload"].startswith("b4_h8_n1024_d64")
    assert bool(d["config"]["causal"]) == causal
    B, H, N, dd = bench.WORKLOADS["b4_h8_n1024_d64"]
    # q, k, v, dO in; o, lse, dq, dk, dv out (bf16 tensors, fp32 lse)
    assert d["e2e"]["h2d_bytes_per_step"] == 4 * B * H * N * dd * 2
    assert d["e2e"]["d2h_bytes_per_step"] == 4 * B * H * N * dd * 2 + B * H * N * 4
    F = bench.fwd_flops(B, H, N, dd, causal)
    assert abs(d["value"] - 3.5 * F / (d["ms_per_step"] * 1e-3) / 1e12) <= 1e-6 * d["value"]


def test_packed_line():
    d = _run("--workload", "varlen_d64_s64_64to1024", "--steps", "3", "--warmup", "3")
    _common(d, 3, 6)
    assert d["config"]["workload"].startswith("varlen_d64_s64_64to1024")
