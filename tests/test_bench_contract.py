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


def test_default_workload_is_the_largest_one_gpu_config():
    sys.path.insert(0, ROOT)
    import bench
    from entropy_active_span_gb300 import workloads as W
    old = sys.argv
    sys.argv = ["bench.py"]
    try:
        a = bench.parse_args()
    finally:
        sys.argv = old
    largest = max((w for w in W.WORKLOADS.values() if w.dtype == "bf16"), key=lambda w: w.T * w.H)
    assert a.workload == largest.name == "long_256k"
    assert a.secondary == "rl_16k"


def test_fractions_use_four_denominators():
    sys.path.insert(0, ROOT)
    import bench
    pk = dict(bf16=2000.0, bf16_sustained=1600.0, hbm=7000.0, source="test")
    f = bench.fractions(1000.0, pk, 1500.0, 152)
    assert abs(f["frac_sustained"] - 1000 / 1600) < 1e-12
    assert abs(f["frac_burst"] - 1000 / 2000) < 1e-12
    assert abs(f["frac_nominal"] - 1000 / 2250) < 1e-12
    assert abs(f["per_clock_peak_tflops"] - 152 * 8192 * 1500e6 / 1e12) < 1e-9
    assert abs(f["frac_per_clock"] - 1000 / f["per_clock_peak_tflops"]) < 1e-12
    assert bench.fractions(1000.0, pk, None, 152)["frac_per_clock"] is None
    # e4m3: every denominator doubles
    f2 = bench.fractions(1000.0, pk, 1500.0, 152, peak_scale=2.0)
    assert abs(f2["frac_per_clock"] - f["frac_per_clock"] / 2) < 1e-12


def test_traffic_is_keyed_by_kernel_build_and_launch_shape():
    sys.path.insert(0, ROOT)
    import bench
    sha = bench.source_sha()
    # a record exists only for the shapes that were captured, never reused for others
    got, src = bench.recorded_traffic("bwd_chunk_gemm_tc", "no_such_workload/c16384")
    assert got is None and src is None
    for path in os.listdir(os.path.join(ROOT, "profiles")):
        for line in open(os.path.join(ROOT, "profiles", path)):
            parts = line.split()
            if parts[:1] == ["traffic"]:
                assert len(parts) == 5 and "/c" in parts[2] and int(parts[3]) > 0
                if parts[4] == sha:
                    assert bench.recorded_traffic(parts[1], parts[2])[0] == int(parts[3])


@pytest.mark.gpu
def test_own_arm_line():
    (d,) = run_bench(["--workload", "rl_4k_v32k", "--steps", "3", "--warmup", "3",
                      "--no-dense", "--no-cpu-baseline", "--secondary", "none"])
    for k in BASE_KEYS + ("roofline", "clocks", "gpu_launches", "phases", "forward_only"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["scaling"] == "weak" and d["dtype"] == "bf16"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert abs(rf["frac_burst"] - rf["achieved"] / rf["peak_burst"]) < 1e-9
    assert abs(rf["frac_nominal"] - rf["achieved"] / 2250.0) < 1e-9
    if d["clocks"]:
        assert rf["frac_per_clock"] > 0 and rf["sm_mhz_median"] == d["clocks"]["sm_mhz"]
    # no ncu capture was made at this shape: the traffic must be null
    assert "traffic" in rf and rf["traffic"] is None
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    c = d["clocks"]
    for k in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert k in c, k
    assert d["gpu_launches"] > 0
    p = d["phases"]
    assert abs(p["spans_ms"] + p["fwd_ms"] + p["bwd_ms"] - d["ms_per_step"]) < 0.1 * d["ms_per_step"]


def test_clock_median_counts_samples_under_load_only(tmp_path):
    """The sampler starts before the warm-up, so its first sample can be
    idle; the median clock and power come from samples under load, and from
    the timed region alone when it holds enough samples."""
    sys.path.insert(0, ROOT)
    import datetime
    import bench

    class Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            pass

    def run(lines, window=None):
        c = bench.ClockSampler.__new__(bench.ClockSampler)
        c.path = str(tmp_path / "clocks.csv")
        open(c.path, "w").write("\n".join(lines) + "\n")
        c.proc = Done()
        c.window = window
        return c.stop()

    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)

    def line(sec, mhz, w, cap="Active"):
        ts = (t0 + datetime.timedelta(seconds=sec)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return (f"{ts}, {mhz}, 2070, {w}, 0x4, Not Active, Not Active, Not Active, {cap}, "
                "3996, 55")

    lines = [line(0.0, 1995, 180.0, "Not Active"), line(0.2, 1500, 1360.0),
             line(0.4, 1400, 1365.0), line(0.6, 1380, 1370.0), line(0.8, 1390, 1366.0)]
    out = run(lines)
    assert out["sm_mhz"] == 1395 and out["samples"] == 5 and out["samples_used"] == 4
    assert out["reasons"] == ["sw_power_cap"] and out["power_w_median"] == 1365.5
    # the timed region holds the last three samples: the warm-up's 1500 MHz drops out
    win = (t0 + datetime.timedelta(seconds=0.3), t0 + datetime.timedelta(seconds=0.9))
    out = run(lines, win)
    assert out["sm_mhz"] == 1390 and out["samples_used"] == 3 and out["basis"].startswith("timed")
