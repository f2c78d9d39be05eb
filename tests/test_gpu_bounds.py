"""The index-checked build on the GPU: small GEMM, attention and encoder shapes (ragged rows,
ragged key tiles, split keys, CTA pairs and single CTAs, half-width last waves) run with every
index check live; the device error word stays clear and every output is bit-equal to the normal
build's. Each build runs in a process of its own (the binding loads one library per process)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu

CHILD = r"""
import json, sys
import numpy as np
import torch
sys.path.insert(0, %(root)r)
sys.path.insert(0, %(root)r + "/tests")
import synth
import transformer_encoder_gb300 as w
from helpers import make_encoder
assert w.lib_path.endswith(%(lib)r), w.lib_path
res = {}
rng = np.random.default_rng(5)
for (M, N, K) in ((1537, 1152, 384), (1, 256, 64), (3000, 1280, 1280), (300, 384, 1536)):
    a = torch.from_numpy(synth.round_to_bf16(rng.standard_normal((M, K)).astype(np.float32))).cuda().to(torch.bfloat16)
    wt = torch.from_numpy(synth.round_to_bf16((0.05 * rng.standard_normal((N, K))).astype(np.float32))).cuda().to(torch.bfloat16)
    b = torch.from_numpy((0.1 * rng.standard_normal(N)).astype(np.float32)).cuda()
    r = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32)).cuda()
    for epi in (0, 1, 2):
        out = w.linear(a, wt, b, epi, resid=r.clone() if epi == 2 else None)
        w.sync_status()
        res[f"linear_{M}_{N}_{K}_{epi}"] = out.float().sum().item()
        res[f"linear_{M}_{N}_{K}_{epi}_bits"] = int(out.view(torch.int16 if out.dtype == torch.bfloat16 else torch.int32).long().sum().item())
for (B, T, H) in ((1, 1, 2), (2, 130, 3), (1, 700, 6), (3, 1500, 4)):
    q, k, v = (torch.randn(B, T, H, 64, device="cuda").to(torch.bfloat16) for _ in range(3))
    out = w.attention(q, k, v)
    w.sync_status()
    res[f"attn_{B}_{T}_{H}"] = int(out.view(torch.int16).long().sum().item())
enc, _, _, g = make_encoder(synth.WORKLOADS["tiny_stack"], keep_host_layers=False)
x = torch.from_numpy(synth.make_input(synth.WORKLOADS["tiny_stack"], g)).cuda()
y = enc.forward(x)
enc.sync_status()
res["tiny_stack"] = int(y.view(torch.int32).long().sum().item())
enc.close()
print(json.dumps(res))
"""


def _run(lib):
    env = dict(os.environ, WENC_LIBRARY=lib)
    torch_seed = "torch.manual_seed(7)\n"
    code = CHILD % {"root": ROOT, "lib": lib}
    code = code.replace("res = {}\n", "res = {}\n" + torch_seed, 1)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_index_checked_build_runs_clean_and_bit_equal():
    from transformer_encoder_gb300.build import build
    build()
    build(bounds_check=True)
    normal = _run("libwenc.so")
    checked = _run("libwenc_bounds.so")
    assert normal.keys() == checked.keys()
    for k in normal:
        assert normal[k] == checked[k], k
