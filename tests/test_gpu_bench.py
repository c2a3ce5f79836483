"""bench.py's default run on the GPU prints one JSON line with the contract's keys:
the metric, whole-job value, roofline of the dominant kernel, cpu_baseline, e2e,
clocks, the library's launch count, and the te.Linear layer and the MXFP8 MLP
measured beside."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_default_bench_line_carries_the_contract():
    out = subprocess.run([sys.executable, "bench.py", "--steps", "3", "--warmup", "3"], cwd=ROOT,
                         capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["scaling"] == "weak"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # value is the step's GEMM FLOPs over the device-timed step
    assert abs(d["value"] - bench.step_flops(bench.WORKLOADS["ln_mlp"]) / (d["ms_per_step"] * 1e-3) / 1e12) \
        <= 1e-3 * d["value"] + 0.01
    assert d["config"]["workload"] == "ln_mlp" and "flushed" in d["config"]["l2"]
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] > 0 and r["achieved"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert r["traffic"] is None or r["traffic"] > 0
    # the FP8 denominator is the larger burst figure: 2 x the measured bf16 burst, or cuBLASLt's FP8
    p = d["fp8_peak"]
    assert r["peak"] == p["used"] == max([p["bf16_burst_x2"]] + list(p["scaled_mm"].values()))
    assert set(d["config"]) == {"workload", "desc", "tokens", "l2", "parallelism"} and d["launch"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 14 * d["steps"]  # the library's kernels of one LayerNormMLP step
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    # the cycle counters' mean SM clock over the timed steps, and the GEMM fraction at that clock
    assert 200 < d["clocks"]["sm_mhz_cycles"] <= 2300
    assert abs(r["frac_at_clock"] - r["frac"] * d["clocks"]["sm_max_mhz"] / d["clocks"]["sm_mhz_cycles"]) < 2e-3
    t = d["te_linear"]
    assert t["workload"] == "linear_hybrid" and t["value"] > 0 and t["gpu_launches"] > 0 and t["e2e"]["value"] > 0
    mx = d["mx_mlp"]
    assert mx["workload"] == "mx_mlp" and mx["value"] > 0 and mx["e2e"]["value"] > 0
    assert abs(mx["value"] - bench.step_flops(bench.WORKLOADS["mx_mlp"]) / (mx["ms_per_step"] * 1e-3) / 1e12) \
        <= 1e-3 * mx["value"] + 0.01
    assert mx["roofline"]["kernel"] == "mxfp8_gemm" and mx["roofline"]["peak"] == r["peak"]
    assert mx["roofline"]["gemm_launches_per_step"] == 6
    assert 0 < mx["quantize"]["frac"] < 1.2 and mx["quantize"]["launches_per_step"] > 0
