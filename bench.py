#!/usr/bin/env python
"""Throughput of the Whisper encoder stack on GB300: 30 s windows per second and TFLOP/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload large_stack] [--impl wenc|reference]
                    [--precision bf16|tf32]

A step is one wenc_forward call over one batch of synthetic windows (all blocks + the final
LayerNorm). Default workload: the large-dims stack (32 blocks, batch 16, T 1500, d 1280,
20 heads x 64, ffn 5120). Weights and inputs are seeded synthetic tensors (no checkpoint).
`value` is windows/s with the input already in HBM, timed over K steps with nothing armed but
the library's launches; the per-kernel times (`kernels`, `roofline`) come from a second pass of
the same K steps with the library's per-launch CUDA events armed. `e2e` is the same metric
through the same C-ABI call with the input copied from pinned host memory and the output copied
back inside the timed region. After the headline (one GPU, default workload) the line also
carries `attention_sweep` (wenc_attention alone at B 16, H 20, T 256 / 1500 / 3000) and
`configs` (the tiny block and the tiny, base and small stacks), each from CUDA events with the
L2 flushed between calls; `--no-extras` skips both. Multi-GPU runs are independent replicas (windows are independent;
there is no collective on the data path): value = all ranks' windows / the slowest rank's time.

`--stem` makes a step the whole encoder from log-mel frames (wenc_encode: the convolutional stem,
the blocks and the final LayerNorm) with the input [B, 3000, n_mels] on the device.

`--cross-kv` adds to each step the decoder's cross-attention K/V precompute over the encoder
output (wenc_cross_kv: 2 x n_layers decoder projections, one GEMM); `e2e` still reads back the
encoder output, not the K/V planes, which a decoder consumes on the device.

`--precision tf32` runs the same step with TF32 tensor-core operands and fp32 activations; its
roofline peak is the measured bf16 peak times the nominal TF32/BF16 ratio (1.1 / 2.25 PFLOP/s).

`--impl reference` times the f64 CPU oracle (the only other implementation) on the host
cores on a bounded sample of the same workload (one block of one window per step, plus that
window's stem with `--stem` and two decoder layers' cross K/V with `--cross-kv`) and
extrapolates to windows/s.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "encoder 30s-windows/sec and TFLOP/s (% of BF16 peak) at 1 GB300"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TF32_PER_BF16 = 1.1 / 2.25  # nominal dense tensor-core rates of GB300 (PFLOP/s)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


# The source files each profiled kernel is built from (plus the shared headers). A traffic
# figure is reported only while these files are byte-identical to the profiled ones.
KERNEL_SOURCES = {
    "gemm": ("gemm.cu",),
    "attention": ("attn.cu",),
    "attention_tf32": ("attn_tf32.cu",),
    "layernorm": ("ln.cu",),
}
SHARED_SOURCES = ("ptx.cuh", "launch.h")


def kernel_source_hash(kernel: str) -> str:
    """sha256 over the CUDA sources of one kernel family and the shared device headers."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "transformer_encoder_gb300", "csrc")
    for name in (*KERNEL_SOURCES[kernel], *SHARED_SOURCES):
        h.update(name.encode())
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _family(launch_name: str, tf32: bool) -> str:
    if launch_name.startswith("gemm_"):
        return "gemm"
    if launch_name == "attention":
        return "attention_tf32" if tf32 else "attention"
    return "layernorm"


def load_traffic(tf32: bool = False):
    """DRAM bytes per launch measured by ncu (profiles/traffic.json), for the launches whose
    kernel sources are still the ones that were profiled; {} when none are."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return {}
    with open(p) as f:
        d = json.load(f)
    hashes = d.get("source_sha256", {})
    per = d.get("bytes_per_launch_tf32" if tf32 else "bytes_per_launch", {})
    return {k: v for k, v in per.items()
            if hashes.get(_family(k, tf32)) == kernel_source_hash(_family(k, tf32))}


def combine_rank_timings(ms_total: float, ms_e2e: float, world: int, device="cuda"):
    """The slowest rank sets the job's time: max over ranks of both timed regions."""
    if world == 1:
        return ms_total, ms_e2e
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms_total, ms_e2e], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0]), float(t[1])


def job_throughput(windows_per_rank: int, world: int, steps: int, ms_total: float) -> float:
    """Windows per second of the whole job: every rank's windows over the slowest rank's time."""
    return windows_per_rank * world * steps / (ms_total / 1e3)


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))


def workload_desc(w):
    return (f"{w.name}: {w.n_layers} blocks, B={w.batch} windows, T={w.seq_len}, d={w.d_model}, "
            f"{w.n_heads} heads x {w.head_dim}, ffn {w.ffn_dim}, final LN {'on' if w.final_ln else 'off'}")


# ------------------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.dev = device_index

    def start(self):
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            target = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            target = str(self.dev)
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", target, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------ CPU oracle
def time_oracle_block(w, seconds: float, steps: int | None = None):
    """Time the f64 oracle on one block of one window; returns (seconds per block, reps)."""
    import numpy as np

    import oracle
    import synth
    rng = np.random.Generator(np.random.PCG64(w.seed))
    p = synth.make_layer(rng, w.d_model, w.ffn_dim, w.bf16_weights)
    x = rng.standard_normal((w.seq_len, w.d_model), dtype=np.float32)
    times = []
    t_end = time.perf_counter() + seconds
    while True:
        t0 = time.perf_counter()
        oracle.encoder_block(x, p, w.n_heads)
        times.append(time.perf_counter() - t0)
        if steps is not None and len(times) >= steps:
            break
        if steps is None and time.perf_counter() >= t_end:
            break
    return times


def time_oracle_stem(w, steps: int):
    """Time the f64 oracle's convolutional stem on one window; returns the per-run seconds."""
    import oracle
    import synth
    p = synth.make_stem(w)
    mel = synth.make_mel(w, batch=1)[0]
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.conv_stem(mel, p["conv1_w"], p["conv1_b"], p["conv2_w"], p["conv2_b"], p["positions"])
        times.append(time.perf_counter() - t0)
    return times


def stem_flops(w) -> float:
    """Dense FLOPs of the stem per call: conv1 (2T x d x 3 n_mels) and conv2 (T x d x 3d)."""
    d, T = w.d_model, w.seq_len
    return 2.0 * w.batch * (2 * T * d * 3 * w.n_mels + T * d * 3 * d)


def time_oracle_cross(w, n_dec: int = 2):
    """Seconds of the f64 oracle's cross K/V precompute for one window and n_dec decoder layers."""
    import numpy as np

    import oracle
    import synth
    dec = synth.make_cross(w, n_dec)
    x = np.random.default_rng(0).standard_normal((w.seq_len, w.d_model))
    t0 = time.perf_counter()
    oracle.cross_kv(x, [p["wk"] for p in dec], [p["wv"] for p in dec], [p["bv"] for p in dec])
    return time.perf_counter() - t0


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform's machine name)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


_ONE_THREAD_ENV = {"OPENBLAS_NUM_THREADS": "1", "OMP_NUM_THREADS": "1", "MKL_NUM_THREADS": "1",
                   "BLIS_NUM_THREADS": "1", "VECLIB_MAXIMUM_THREADS": "1", "NUMEXPR_NUM_THREADS": "1"}


def time_oracle_block_single_thread(w, runs: int = 2, timeout: float = 120.0):
    """Seconds per block of the f64 oracle with one BLAS thread (a child process, since the BLAS
    thread count is fixed when numpy loads); None if the child fails or runs out of time."""
    code = ("import json, sys; sys.path.insert(0, %r); import bench, synth; "
            "print(json.dumps(bench.time_oracle_block(synth.WORKLOADS[%r], 0.0, steps=%d)))" % (ROOT, w.name, runs))
    env = dict(os.environ, **_ONE_THREAD_ENV)
    try:
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=timeout)
        return statistics.median(json.loads(r.stdout.strip().splitlines()[-1])) if r.returncode == 0 else None
    except Exception:
        return None


def cpu_baseline(w, seconds: float, with_stem: bool = False, with_cross: bool = False, single_thread: bool = True):
    times = time_oracle_block(w, seconds)
    t_block = statistics.median(times)
    t_stem = statistics.median(time_oracle_stem(w, 3)) if with_stem else 0.0
    t_cross = time_oracle_cross(w, 2) * w.n_layers / 2 if with_cross else 0.0
    win_s = 1.0 / (t_block * w.n_layers + t_stem + t_cross)
    stem_note = f" + the stem ({t_stem:.3f} s, median of 3)" if with_stem else ""
    if with_cross:
        stem_note += f" + cross K/V of 2 decoder layers x{w.n_layers / 2:g} ({t_cross:.3f} s)"
    line = {"value": win_s, "unit": "windows/s", "cores": host_cores(), "kind": "oracle",
            "sample": (f"f64 numpy oracle, one block of one {w.seq_len}-frame window at {w.name} dims, "
                       f"median of {len(times)} runs ({t_block:.3f} s/block), extrapolated x{w.n_layers} blocks"
                       + stem_note + "; all cores (BLAS threads = host cores)"),
            "seconds_per_block": t_block, "cpu_model": cpu_model(), "nproc": os.cpu_count()}
    if single_thread:
        t1 = time_oracle_block_single_thread(w)
        line["single_thread"] = (None if t1 is None else
                                 {"value": 1.0 / (t1 * w.n_layers + t_stem + t_cross), "unit": "windows/s",
                                  "cores": 1, "seconds_per_block": t1,
                                  "sample": "the same block with one BLAS thread (median of 2 runs), extrapolated "
                                            f"x{w.n_layers} blocks" + (" (stem and cross K/V at all cores)"
                                                                       if with_stem or with_cross else "")})
    return line


# ------------------------------------------------------------------------------------------ arms
def run_reference(args, w):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    # Each step: one block of one window (x n_layers), plus, with --stem, the stem of that window
    # and, with --cross-kv, the cross K/V of two decoder layers (x n_layers / 2): the work of one
    # window of the wenc arm's step, extrapolated from a bounded sample.
    def step_seconds():
        t = time_oracle_block(w, 0.0, steps=1)[0] * w.n_layers
        if args.stem:
            t += time_oracle_stem(w, 1)[0]
        if args.cross_kv:
            t += time_oracle_cross(w, 2) * w.n_layers / 2
        return t

    for _ in range(args.warmup):  # warm-up (untimed)
        step_seconds()
    total = sum(step_seconds() for _ in range(args.steps))
    win_s = args.steps / total
    extra = (" + the convolutional stem" if args.stem else "") + \
            (f" + cross K/V of 2 decoder layers x{w.n_layers / 2:g}" if args.cross_kv else "")
    sample = f"one block of one window per step at {w.name} dims, x{w.n_layers} blocks{extra}"
    line = {
        "impl": "reference", "metric": METRIC, "value": win_s, "unit": "windows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(w) + extra, "sample": sample + ", extrapolated"},
        "cpu_baseline": {"value": win_s, "unit": "windows/s", "cores": host_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": win_s, "unit": "windows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def build_encoder(w, precision: str = "bf16"):
    """The library's encoder over workload w's seeded synthetic weights; returns (encoder, the
    generator positioned after the weights, from which the input is drawn)."""
    import torch

    import synth
    from transformer_encoder_gb300 import Encoder
    dev_layers = []

    def up(p):
        out = {}
        for k, v in p.items():
            t = torch.from_numpy(v)
            if k in synth.MATRIX_KEYS and w.bf16_weights:
                t = t.to(torch.bfloat16)
            out[k] = t.cuda()
        return out

    _, final, rng = synth.make_weights(w, layer_callback=lambda p: dev_layers.append(up(p)))
    fin = (torch.from_numpy(final[0]).cuda(), torch.from_numpy(final[1]).cuda()) if w.final_ln else None
    enc = Encoder(dev_layers, w.n_heads, w.seq_len, w.batch, final=fin, precision=precision)
    del dev_layers
    torch.cuda.empty_cache()
    return enc, rng


def _l2_flush_buffer():
    import torch
    return torch.empty(64 << 20, dtype=torch.float32, device="cuda")  # 256 MB, twice the L2


def attention_sweep(peaks, reps: int = 10):
    """wenc_attention alone at B = 16, H = 20, hd = 64 for T in {256, 1500, 3000}: median CUDA-event
    time per call (L2 flushed before each), TFLOP/s and fraction of the measured bf16 burst peak."""
    import torch

    from transformer_encoder_gb300 import attention, sync_status
    B, H = 16, 20
    flush = _l2_flush_buffer()
    gen = torch.Generator(device="cuda").manual_seed(1)
    res = {}
    for T in (256, 1500, 3000):
        q, k, v = (torch.randn(B, T, H, 64, device="cuda", generator=gen).to(torch.bfloat16) for _ in range(3))
        out = torch.empty_like(q)
        for _ in range(3):
            attention(q, k, v, out)
        evs = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            attention(q, k, v, out)
            e1.record()
            evs.append((e0, e1))
        torch.cuda.synchronize()
        sync_status()
        us = 1e3 * statistics.median(a.elapsed_time(b) for a, b in evs)
        tf = 4.0 * B * H * T * T * 64 / (us * 1e-6) / 1e12
        res[str(T)] = {"B": B, "H": H, "hd": 64, "us": us, "tflops": tf, "frac_of_bf16_burst": tf / peaks["bf16_tflops"],
                       "launches": 1, "inputs": "q, k, v ~ N(0, 1) bf16 [B, T, H, 64], seed 1; L2 flushed before each call"}
        del q, k, v, out
    return res


def configs_throughput(peaks, steps: int = 20, warmup: int = 3):
    """The four smaller workloads (tiny block, tiny, base and small stacks): windows/s and TFLOP/s of
    wenc_forward from CUDA events around each step, with the L2 flushed between steps (their
    weights and activations would otherwise stay in the 126 MB L2)."""
    import torch

    import synth
    res = {}
    flush = _l2_flush_buffer()
    for name in ("tiny_block", "tiny_stack", "base_stack", "small_stack"):
        w = synth.WORKLOADS[name]
        enc, rng = build_encoder(w)
        x = torch.from_numpy(synth.make_input(w, rng)).cuda()
        out = torch.empty_like(x)
        for _ in range(warmup):
            enc.forward(x, out)
        evs = []
        for _ in range(steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            enc.forward(x, out)
            e1.record()
            evs.append((e0, e1))
        torch.cuda.synchronize()
        enc.sync_status()
        ms = sum(a.elapsed_time(b) for a, b in evs)
        tf = w.flops() * steps / (ms / 1e3) / 1e12
        res[name] = {"workload": workload_desc(w), "windows_per_s": w.batch * steps / (ms / 1e3),
                     "ms_per_step": ms / steps, "tflops": tf, "frac_of_bf16_burst": tf / peaks["bf16_tflops"],
                     "launches_per_step": enc.launches(),
                     "bound": ("latency: a forward this small is a few dozen microseconds of dependent launches"
                               if w.flops() < 0.1e12 else "tensor (GEMMs) with latency at the launch boundaries"),
                     "weights": "f32 (rounded to bf16 at create)" if not w.bf16_weights else "bf16"}
        enc.close()
        del x, out
        torch.cuda.empty_cache()
    return res


def run_wenc(args, w):
    import numpy as np
    import torch

    import synth
    from transformer_encoder_gb300 import LAUNCH_KINDS

    rank, local_rank, world = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the wenc path has no CPU fallback)")
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    peaks, peak_src = load_peaks()

    # ---- weights and inputs (seeded synthetic; identical on every rank)
    enc, rng = build_encoder(w, args.precision)
    tf32 = args.precision == "tf32"
    if args.stem:
        stem = synth.make_stem(w)
        enc.set_stem({k: (torch.from_numpy(v).to(torch.bfloat16) if k in ("conv1_w", "conv2_w") and w.bf16_weights
                          else torch.from_numpy(v)).cuda() for k, v in stem.items()})
        x_host = torch.from_numpy(synth.make_mel(w)).pin_memory()
        step = enc.encode
        n_launch = enc.encode_launches()
    else:
        x_host = torch.from_numpy(synth.make_input(w, rng)).pin_memory()
        step = enc.forward
        n_launch = enc.launches()
    if args.cross_kv:
        mdt = torch.bfloat16 if w.bf16_weights else torch.float32
        enc.set_cross_kv([{"wk": torch.from_numpy(p["wk"]).to(mdt).cuda(), "wv": torch.from_numpy(p["wv"]).to(mdt).cuda(),
                           "bv": torch.from_numpy(p["bv"]).cuda()} for p in synth.make_cross(w)])
        kv = torch.empty((2 * w.n_layers, w.batch * w.seq_len, w.d_model),
                         dtype=torch.float32 if tf32 else torch.bfloat16, device="cuda")
        base_step = step
        n_base = n_launch

        def step(x_, out_):
            base_step(x_, out_)
            enc.cross_kv(out_, kv)
        n_launch += 2
    x = x_host.cuda()
    out = torch.empty((w.batch, w.seq_len, w.d_model), dtype=torch.float32, device="cuda")
    out_host = torch.empty(tuple(out.shape), dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        step(x, out)
    torch.cuda.synchronize()
    enc.sync_status()

    # ---- timed region (the headline): K steps with nothing armed but the library's own launches
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    step_ev[0].record(stream)
    for k in range(args.steps):
        step(x, out)
        step_ev[k + 1].record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms_total = step_ev[0].elapsed_time(step_ev[-1])
    step_ms = sorted(step_ev[k].elapsed_time(step_ev[k + 1]) for k in range(args.steps))

    def pct(q):
        return step_ms[min(len(step_ms) - 1, int(round(q * (len(step_ms) - 1))))]
    enc.sync_status()

    # ---- per-kernel breakdown: a second pass of K steps with the library's per-launch events armed
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_launch + 1)] for _ in range(args.steps)]
    for row in ev:  # torch creates the CUDA event on its first record; the library needs real handles
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    kinds = None
    k_start = torch.cuda.Event(enable_timing=True)
    k_stop = torch.cuda.Event(enable_timing=True)
    k_start.record(stream)
    for k in range(args.steps):
        if args.cross_kv:
            # the timing hook covers one library call: arm it for the encoder, then for the
            # cross K/V call (whose first event repeats the encoder's last one)
            ks1 = enc.set_launch_events(ev[k][:n_base + 1])
            base_step(x, out)
            ks2 = enc.set_launch_events(ev[k][n_base:])
            enc.cross_kv(out, kv)
            ks = list(ks1)[:n_base] + list(ks2)[:2]
        else:
            ks = enc.set_launch_events(ev[k])
            step(x, out)
        if kinds is None:
            kinds = ks
    k_stop.record(stream)
    torch.cuda.synchronize()
    ms_hooked = k_start.elapsed_time(k_stop)
    enc.sync_status()

    # per-kind device time over the timed region
    per_kind = {}
    for k in range(args.steps):
        for i in range(n_launch):
            name = LAUNCH_KINDS[kinds[i]]
            per_kind.setdefault(name, [0.0, 0])
            per_kind[name][0] += ev[k][i].elapsed_time(ev[k][i + 1])
            per_kind[name][1] += 1

    # ---- e2e through the same call with host buffers: every step copies its input from pinned
    # host memory and reads its result back inside the timed region. The copies run on a stream
    # of their own with two device buffer pairs, so step k+1's upload and step k's readback
    # overlap the encoder's work, as a pipelined caller would run it; events order every reuse.
    copy_stream = torch.cuda.Stream()
    xs = [x, torch.empty_like(x)]
    outs = [out, torch.empty_like(out)]
    outs_host = [out_host, torch.empty_like(out_host).pin_memory()]
    ev_h2d = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_d2h = [torch.cuda.Event() for _ in range(2)]
    for e_ in ev_done + ev_d2h:
        e_.record(stream)

    def e2e_steps(n):
        def h2d(k):  # step k's input into xs[k % 2], once step k-2 has finished reading it
            i = k & 1
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(ev_done[i])
                xs[i].copy_(x_host, non_blocking=True)
                ev_h2d[i].record(copy_stream)

        h2d(0)
        for k in range(n):
            i = k & 1
            if k + 1 < n:
                h2d(k + 1)  # enqueued ahead of step k's readback: it runs during step k
            stream.wait_event(ev_h2d[i])
            stream.wait_event(ev_d2h[i])  # step k-2's result has been read out of outs[i]
            step(xs[i], outs[i])
            ev_done[i].record(stream)
            with torch.cuda.stream(copy_stream):  # runs during step k+1
                copy_stream.wait_event(ev_done[i])
                outs_host[i].copy_(outs[i], non_blocking=True)
                ev_d2h[i].record(copy_stream)
        for i in range(2):
            stream.wait_event(ev_d2h[i])

    e2e_steps(2)
    torch.cuda.synchronize()
    barrier()
    e_start = torch.cuda.Event(enable_timing=True)
    e_stop = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    copy_stream.wait_event(e_start)
    e2e_steps(args.steps)
    e_stop.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms_e2e = e_start.elapsed_time(e_stop)

    # The host link alone, outside the timed regions: one upload and one readback of a step's
    # buffers on the copy stream (explains the part of e2e that the copies cannot overlap: the
    # first upload and the last readback of the timed region).
    def copy_ms(dst, src):
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(copy_stream):
            c0.record(copy_stream)
            dst.copy_(src, non_blocking=True)
            c1.record(copy_stream)
        torch.cuda.synchronize()
        return c0.elapsed_time(c1)
    h2d_ms = min(copy_ms(xs[0], x_host) for _ in range(3))
    d2h_ms = min(copy_ms(outs_host[0], outs[0]) for _ in range(3))

    ms_total, ms_e2e = combine_rank_timings(ms_total, ms_e2e, world)

    ms_step = ms_total / args.steps
    windows = w.batch * world
    value = job_throughput(w.batch, world, args.steps, ms_total)
    cross_flops = 2.0 * w.batch * w.seq_len * (2 * w.n_layers * w.d_model) * w.d_model
    flops_step = w.flops() + (stem_flops(w) if args.stem else 0.0) + (cross_flops if args.cross_kv else 0.0)
    tflops = flops_step * world / (ms_step / 1e3) / 1e12

    # ---- roofline of the dominant kernel (the tcgen05 GEMM: four launches per block)
    M, d, f, T, H = w.rows, w.d_model, w.ffn_dim, w.seq_len, w.n_heads
    gemm_flops = {"gemm_qkv": 2.0 * M * 3 * d * d, "gemm_out": 2.0 * M * d * d,
                  "gemm_fc1": 2.0 * M * f * d, "gemm_fc2": 2.0 * M * d * f}
    attn_flops = 4.0 * w.batch * H * T * T * w.head_dim
    ln_bytes = (8.0 if tf32 else 6.0) * M * d  # fp32 read + bf16 or fp32 write
    es = 4 if tf32 else 2
    kp1 = (3 * w.n_mels + 63) // 64 * 64
    stem_gemm_flops = {"gemm_conv1": 2.0 * w.batch * 2 * T * d * 3 * w.n_mels,
                       "gemm_conv2": 2.0 * w.batch * T * d * 3 * d}
    # both unfold launches of a step: read the signal, write the unfolded rows
    unfold_bytes = (w.batch * 2 * T * (w.n_mels * 4 + kp1 * es)) + (w.batch * (2 * T * d * es + T * 3 * d * es))
    kern = {}
    for name, (ms, n) in per_kind.items():
        avg = ms / n
        if name in gemm_flops:
            kern[name] = {"launches": n, "avg_us": 1e3 * avg, "tflops": gemm_flops[name] / (avg / 1e3) / 1e12}
        elif name == "attention":
            kern[name] = {"launches": n, "avg_us": 1e3 * avg, "tflops": attn_flops / (avg / 1e3) / 1e12}
        elif name in stem_gemm_flops:
            kern[name] = {"launches": n, "avg_us": 1e3 * avg, "tflops": stem_gemm_flops[name] / (avg / 1e3) / 1e12}
        elif name == "gemm_cross_kv":
            kern[name] = {"launches": n, "avg_us": 1e3 * avg, "tflops": cross_flops / (avg / 1e3) / 1e12}
        elif name == "cross_kv_cast":
            kern[name] = {"launches": n, "avg_us": 1e3 * avg, "gbs": M * d * (4 + es) / (avg / 1e3) / 1e9}
        elif name == "row_stats":
            kern[name] = {"launches": n, "avg_us": 1e3 * avg, "gbs": 6.0 * M * d / (avg / 1e3) / 1e9}
        elif name == "stem_unfold":
            kern[name] = {"launches": n, "avg_us": 1e3 * avg, "gbs": unfold_bytes * args.steps / (ms / 1e3) / 1e9}
        elif name in ("layernorm", "layernorm_final"):
            b = ln_bytes if name == "layernorm" else 8.0 * M * d
            kern[name] = {"launches": n, "avg_us": 1e3 * avg, "gbs": b / (avg / 1e3) / 1e9}
        else:
            kern[name] = {"launches": n, "avg_us": 1e3 * avg}
        kern[name]["share"] = ms / sum(v[0] for v in per_kind.values())
    g_ms = sum(per_kind[k][0] for k in gemm_flops if k in per_kind)
    g_n = sum(per_kind[k][1] for k in gemm_flops if k in per_kind)
    g_flops_per_launch = sum(gemm_flops[k] * per_kind[k][1] for k in gemm_flops if k in per_kind) / g_n
    g_achieved = g_flops_per_launch / (g_ms / g_n / 1e3) / 1e12
    peak = peaks.get("bf16_tflops_sustained", PEAKS_FALLBACK["bf16_tflops_sustained"])
    peak_name = "bf16_tflops_sustained"
    if tf32:
        peak *= TF32_PER_BF16
        peak_name = "bf16_tflops_sustained x 1.1/2.25 (nominal TF32/BF16)"
    per = load_traffic(tf32) if w.name in ("large_stack", "large_block") else {}
    g_traffic = None
    if per:
        for name in kern:
            if name in per:
                kern[name]["traffic_bytes"] = per[name]
        if all(k in per for k in gemm_flops):
            g_traffic = sum(per[k] * per_kind[k][1] for k in gemm_flops) / g_n
    roofline = {"kernel": f"gemm_tc_kernel{' (TF32)' if tf32 else ''} (QKV, out-proj, fc1, fc2 launches)",
                "bound": "tensor", "achieved": g_achieved, "peak": peak, "unit": "TFLOP/s", "frac": g_achieved / peak,
                "peak_source": f"{peak_name}, {peak_src}", "traffic": g_traffic,
                "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)"}

    line = {
        "metric": METRIC, "value": value, "unit": "windows/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "tf32" if tf32 else "bf16", "data": "synthetic",
        "ms_per_step_pct": {"p10": pct(0.1), "p50": pct(0.5), "p90": pct(0.9), "from": "CUDA events between steps"},
        "config": {"workload": workload_desc(w) + (f", from {2 * T} log-mel frames x {w.n_mels} through the "
                                                   "convolutional stem" if args.stem else "")
                   + (f", plus the cross-attention K/V of {w.n_layers} decoder layers (e2e reads back the encoder "
                      "output only)" if args.cross_kv else ""),
                   "windows_per_step": w.batch, "seq_len": T,
                   "l2": "no flush: each step streams 1.26 GB of weights and >400 MB of activations, above the 126 MB L2"
                   if w.name == "large_stack" else "no flush",
                   "parallelism": f"replicas x{world}", "precision": args.precision},
        "tflops": tflops,
        "pct_of_bf16_peak": {"burst": 100 * tflops / world / peaks["bf16_tflops"],
                             "sustained": 100 * tflops / world / peaks["bf16_tflops_sustained"],
                             "source": peak_src},
        "roofline": roofline,
        "kernels": kern,
        "kernels_pass": {"ms_per_step": ms_hooked / args.steps,
                         "note": "the per-kernel times come from a second pass of the same K steps with the "
                                 "library's per-launch CUDA events armed; value and ms_per_step come from a pass "
                                 "without them"},
        "gpu_launches": n_launch * args.steps,
        "e2e": {"value": windows * args.steps / (ms_e2e / 1e3), "unit": "windows/s",
                "h2d_bytes_per_step": x.numel() * 4, "d2h_bytes_per_step": out.numel() * 4,
                "copies": "pinned host memory, on a copy stream overlapping the previous/next step (double-buffered)",
                "h2d_gbs": x.numel() * 4 / (h2d_ms / 1e3) / 1e9, "d2h_gbs": out.numel() * 4 / (d2h_ms / 1e3) / 1e9},
        "clocks": clk,
    }
    enc.close()
    del x, out, xs, outs
    torch.cuda.empty_cache()
    extras = (world == 1 and not args.no_extras and w.name == "large_stack" and not tf32
              and not args.stem and not args.cross_kv)
    if extras:
        line["attention_sweep"] = attention_sweep(peaks)
        line["configs"] = configs_throughput(peaks)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, with_stem=args.stem, with_cross=args.cross_kv)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("wenc", "reference"), default="wenc")
    ap.add_argument("--workload", default="large_stack")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the oracle's CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the standalone attention sweep and the four smaller workloads after the headline")
    ap.add_argument("--cross-kv", action="store_true",
                    help="add the decoder cross-attention K/V precompute over the encoder output to each step")
    ap.add_argument("--stem", action="store_true",
                    help="time the whole encoder from log-mel frames (convolutional stem + blocks)")
    ap.add_argument("--precision", choices=("bf16", "tf32"), default="bf16",
                    help="tensor-core operand precision of the timed path")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "wenc":
        print("note: warm-up raised to the minimum of 3 steps", file=sys.stderr)
        args.warmup = 3
    import synth
    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_wenc(args, w)


if __name__ == "__main__":
    sys.exit(main())
