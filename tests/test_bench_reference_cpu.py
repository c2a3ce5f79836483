"""bench.py --impl reference on the host: the oracle arm's JSON line carries the
contract's keys, our arm's metric and unit, and a cpu_baseline describing the run."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "linear_fwd",
                          "--steps", "3", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "linear_fwd"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and "oracle" in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # each timed step is a sample scaled to a whole step, and the line says so
    assert d["extrapolated"] is True and d["timed_wall_s"] > 0 and d["sampled_ms_per_step"] > 0
    # the config is the GPU arm's, key for key (how that arm launches is a top-level key)
    assert set(d["config"]) == {"workload", "desc", "tokens", "l2", "parallelism"}
