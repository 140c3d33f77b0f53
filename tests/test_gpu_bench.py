"""The GPU arm of bench.py on a small workload: one JSON line with every field the benchmark
line carries (throughput, roofline of the attention kernel, the shift kernel's record, the
end-to-end leg through host memory, the launch count, clocks, the cpu baseline from the
oracle, and the accuracy against it), each with values that are consistent with each
other."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                          text=True, timeout=900)


@pytest.mark.gpu
def test_bench_json_line_small_workload():
    import oracle  # noqa: F401  (builds the oracle's C library before the subprocess uses it)

    r = run_bench("--workload", "kbias20_b1h28g4_s4096_d128_causal", "--steps", "3", "--warmup", "3", "--no-also",
                  "--cpu-budget", "2")
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench

    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["scaling"] == "weak"
    assert d["data"] == "synthetic" and d["dtype"] == "f16"
    assert d["config"]["workload"] == "kbias20_b1h28g4_s4096_d128_causal"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # the step's throughput and its time agree (FLOPs of the workload per step)
    flops = bench.wl.WORKLOADS["kbias20_b1h28g4_s4096_d128_causal"].flops()
    assert abs(d["value"] - flops / (d["ms_per_step"] * 1e-3) / 1e12) <= 1e-3 * d["value"] + 0.1
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s" and rf["peak"] > 0
    assert rf["achieved"] >= d["value"] * 0.999   # the attention kernel alone is at least the step's rate
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    ks = d["kshift"]
    assert ks["bound"] == "hbm" and ks["unit"] == "GB/s" and ks["bytes_per_launch"] > 0 and ks["ms"] > 0
    iso = ks["isolated"]
    assert iso["ms"] > 0 and abs(iso["achieved"] - ks["bytes_per_launch"] / (iso["ms"] * 1e-3) / 1e9) < 1.0
    e2e = d["e2e"]
    assert e2e["unit"] == "TFLOP/s" and 0 < e2e["value"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["max_step_ms"] >= e2e["median_step_ms"] > 0
    assert d["gpu_launches"] > 0
    ck = d["clocks"]
    assert "sm_mhz" in ck and "sm_max_mhz" in ck and isinstance(ck["reasons"], list)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    rm = d["rmse"]
    assert rm["rows"] > 0 and rm["rel_rmse"] is not None and rm["rel_rmse"] < 5e-3
    assert d["finite_output"] is True
