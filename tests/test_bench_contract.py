"""The JSON line bench.py prints: every key the benchmark contract requires,
for the oracle arm (on the CPU) and for the library's own arm (on a GPU, a
reduced workload)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e")


def run_bench(args, env=None, timeout=600):
    e = dict(os.environ)
    e.update(env or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout, env=e)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    return [json.loads(l) for l in lines]


def test_reference_arm_line():
    (d,) = run_bench(["--impl", "reference", "--workload", "tiny_fp32", "--steps", "2",
                      "--warmup", "1"])
    for k in BASE_KEYS:
        assert k in d, k
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 2
    assert d["config"]["workload"] == "tiny_fp32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]


def test_reference_arm_other_ranks_print_nothing():
    assert run_bench(["--impl", "reference", "--workload", "tiny_fp32", "--steps", "1",
                      "--warmup", "1"], env={"RANK": "1", "WORLD_SIZE": "2"}) == []


@pytest.mark.gpu
def test_own_arm_line():
    (d,) = run_bench(["--workload", "rl_4k_v32k", "--steps", "3", "--warmup", "3",
                      "--no-dense", "--no-cpu-baseline"])
    for k in BASE_KEYS + ("roofline", "clocks", "gpu_launches", "phases", "forward_only"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["scaling"] == "weak" and d["dtype"] == "bf16"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert "traffic" in rf
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    c = d["clocks"]
    for k in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert k in c, k
    assert d["gpu_launches"] > 0
    p = d["phases"]
    assert abs(p["spans_ms"] + p["fwd_ms"] + p["bwd_ms"] - d["ms_per_step"]) < 0.1 * d["ms_per_step"]
