"""bench.py's reference arm (the f64 oracle timed on the host cores) prints one JSON line that
keeps the bench contract; under a multi-rank launch only rank 0 runs and prints. CPU only."""
import contextlib
import io
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

ARGS = ["--impl", "reference", "--workload", "tiny_block", "--steps", "1", "--warmup", "1"]


def _run(monkeypatch, rank=None, world=None):
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    if rank is not None:
        monkeypatch.setenv("RANK", str(rank))
        monkeypatch.setenv("LOCAL_RANK", str(rank))
        monkeypatch.setenv("WORLD_SIZE", str(world))
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(ARGS + (["--gpus", str(world)] if world else []))
    return rc, [l for l in buf.getvalue().splitlines() if l.strip()]


def test_reference_line_keeps_the_contract(monkeypatch):
    rc, lines = _run(monkeypatch)
    assert rc == 0 and len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "windows/s" and d["higher_is_better"] is True and d["value"] > 0
    assert (d["steps"], d["warmup"], d["n_gpus"]) == (1, 1, 1)
    assert d["ms_per_step"] > 0 and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "windows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_runs_on_rank_zero_only(monkeypatch):
    rc, lines = _run(monkeypatch, rank=1, world=2)
    assert rc == 0 and lines == []


def test_reference_times_the_stem_and_cross_kv_when_asked(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(ARGS + ["--stem", "--cross-kv"])
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert rc == 0 and len(lines) == 1
    d = json.loads(lines[0])
    assert "stem" in d["config"]["workload"] and "cross K/V" in d["config"]["workload"]
    assert "stem" in d["cpu_baseline"]["sample"] and d["value"] > 0
