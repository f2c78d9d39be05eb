"""bench.py's CPU baseline: the host's CPU model and the single-thread leg (CPU only, no GPU)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_cpu_model_is_named():
    name = bench.cpu_model()
    assert isinstance(name, str) and name.strip()


def test_single_thread_leg_times_one_block():
    w = synth.WORKLOADS["tiny_block"]
    t = bench.time_oracle_block_single_thread(w, runs=1, timeout=300)
    assert t is not None and t > 0


def test_cpu_baseline_carries_both_legs():
    w = synth.WORKLOADS["tiny_block"]
    line = bench.cpu_baseline(w, 0.0)
    assert line["kind"] == "oracle" and line["cores"] >= 1 and line["cpu_model"]
    st = line["single_thread"]
    assert st is not None and st["cores"] == 1 and st["value"] > 0
    assert st["unit"] == line["unit"] == "windows/s"
