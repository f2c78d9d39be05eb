"""Host logic of the multi-GPU bench path on CPU: two gloo ranks, no GPU.

The windows of a batch are independent, so N GPUs run N replicas with no data-path
collective; the only exchange is the max over ranks of the timed regions, which sets the
job's time. This checks that reduction and the whole-job throughput built on it."""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out_q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_total, ms_e2e = bench.combine_rank_timings(100.0 + 50.0 * rank, 200.0 - 10.0 * rank, world, device="cpu")
        value = bench.job_throughput(16, world, 10, ms_total)
        out_q.put((rank, ms_total, ms_e2e, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29000 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms_total, ms_e2e, value in res:
        assert ms_total == 150.0 and ms_e2e == 200.0          # slowest rank, per region
        assert value == pytest.approx(16 * 2 * 10 / 0.150)   # all ranks' windows / slowest time


def test_single_rank_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.combine_rank_timings(12.5, 20.0, 1) == (12.5, 20.0)
    assert bench.job_throughput(16, 1, 20, 1000.0) == pytest.approx(320.0)


def test_traffic_figures_track_the_kernel_sources():
    sys.path.insert(0, ROOT)
    import json

    import bench
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    recorded = d["source_sha256"]
    for tf32, key in ((False, "bytes_per_launch"), (True, "bytes_per_launch_tf32")):
        got = bench.load_traffic(tf32)
        for name in d.get(key, {}):
            fam = bench._family(name, tf32)
            # a figure is reported exactly while its kernel's sources are the profiled ones
            assert (name in got) == (recorded.get(fam) == bench.kernel_source_hash(fam)), (name, tf32)


def test_traffic_gate_drops_a_changed_kernel(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    real = bench.kernel_source_hash
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "changed" if k == "attention" else real(k))
    got = bench.load_traffic(False)
    assert "attention" not in got
