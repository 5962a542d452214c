"""The reference arm of bench.py (the CPU oracle timed on whole 4096x4096 matrices, rows split over
the host's cores) prints one JSON line with the keys of the benchmark contract, and its step time
is what the run actually spent; it needs no GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is False and d["value"] > 0 and d["unit"] == "us/matrix"
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert cb["cores"] == len(os.sched_getaffinity(0))
    # the timed steps are whole matrices: their sum is the timed wall time, not a projection
    assert abs(d["steps"] * d["ms_per_step"] / 1e3 - d["timed_seconds"]) <= 0.05 * d["timed_seconds"] + 0.01
