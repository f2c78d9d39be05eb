"""bench.py's own arm on the GPU keeps the contract the driver reads: one JSON line with the
headline keys, the roofline and clock records, e2e with the copied bytes, the launch count, and,
for the default workload, the attention sweep and the smaller configurations."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


def _line(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_bench_line_keeps_the_contract():
    sys.path.insert(0, ROOT)
    import bench
    d = _line("--workload", "tiny_stack", "--steps", "4", "--warmup", "3", "--no-cpu-baseline")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "clocks", "gpu_launches", "kernels",
                "kernels_pass"):
        assert key in d, key
    assert d["metric"] == bench.METRIC and d["unit"] == "windows/s" and d["value"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 4 and d["warmup"] == 3 and d["dtype"] == "bf16"
    assert d["config"]["workload"].startswith("tiny_stack")
    # tiny stack: 1 row-statistics + 4 blocks x (QKV, attention, merge of split keys, out, LN2, fc1, fc2) + final LN
    assert d["gpu_launches"] == 4 * 30
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s" and 0 < rf["frac"] < 1.5
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    e = d["e2e"]
    assert e["unit"] == "windows/s" and e["value"] > 0
    assert e["h2d_bytes_per_step"] == e["d2h_bytes_per_step"] == 1500 * 384 * 4
    assert e["h2d_gbs"] > 0 and e["d2h_gbs"] > 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    pc = d["ms_per_step_pct"]
    assert pc["p10"] <= pc["p50"] <= pc["p90"] and abs(pc["p50"] - d["ms_per_step"]) < 0.5 * d["ms_per_step"]
    assert "attention_sweep" not in d and "configs" not in d  # only after the default workload's headline


def test_bench_extras_are_well_formed():
    sys.path.insert(0, ROOT)
    import bench
    peaks, _ = bench.load_peaks()
    sweep = bench.attention_sweep(peaks, reps=3)
    assert sorted(sweep, key=int) == ["256", "1500", "3000"]
    for T, v in sweep.items():
        assert v["B"] == 16 and v["H"] == 20 and v["us"] > 0
        assert abs(v["tflops"] - 4.0 * 16 * 20 * int(T) ** 2 * 64 / (v["us"] * 1e-6) / 1e12) < 1e-6 * v["tflops"]
    cfg = bench.configs_throughput(peaks, steps=3, warmup=3)
    assert list(cfg) == ["tiny_block", "tiny_stack", "base_stack", "small_stack"]
    for v in cfg.values():
        assert v["windows_per_s"] > 0 and v["tflops"] > 0 and 0 < v["frac_of_bf16_burst"] < 1.5
