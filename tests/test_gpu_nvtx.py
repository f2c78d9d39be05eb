"""The optional NVTX ranges (WENC_NVTX=1) change nothing the library computes: a forward of the
tiny stack run with them is bit-equal to one run without (each in a process of its own, since
the switch is read once)."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu

CHILD = r"""
import sys, hashlib
sys.path.insert(0, %(root)r); sys.path.insert(0, %(root)r + "/tests")
import torch, synth
from helpers import make_encoder
w = synth.WORKLOADS["tiny_stack"]
enc, _, _, rng = make_encoder(w, keep_host_layers=False)
x = torch.from_numpy(synth.make_input(w, rng)).cuda()
y = enc.forward(x)
enc.sync_status()
print(hashlib.sha256(y.cpu().numpy().tobytes()).hexdigest())
"""


def _run(nvtx: bool):
    env = dict(os.environ)
    env.pop("WENC_NVTX", None)
    if nvtx:
        env["WENC_NVTX"] = "1"
    r = subprocess.run([sys.executable, "-c", CHILD % {"root": ROOT}], capture_output=True, text=True, env=env,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    return r.stdout.strip().splitlines()[-1]


def test_nvtx_ranges_leave_results_unchanged():
    assert _run(True) == _run(False)
