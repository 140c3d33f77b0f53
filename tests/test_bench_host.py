"""Host-only checks of bench.py: the reference arm (the fp64 CPU oracle) prints one JSON
line with the fields the benchmark contract names, and a non-zero rank prints nothing."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=e,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_json_line():
    import oracle  # noqa: F401  (builds the oracle's C library once, before the subprocess)

    r = run_bench("--impl", "reference", "--workload", "iid_b1h1_s128_d64", "--steps", "2", "--warmup", "1",
                  "--cpu-budget", "2")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    import bench

    assert d["metric"] == bench.METRIC     # the GPU arm prints the same metric, so the two compare
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["config"]["workload"] == "iid_b1h1_s128_d64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing():
    r = run_bench("--impl", "reference", "--workload", "iid_b1h1_s128_d64", "--steps", "1", "--warmup", "0",
                  "--cpu-budget", "1", env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
