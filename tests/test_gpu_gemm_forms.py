"""The two forms of the bf16 256-column GEMM give the same bits.

By default those GEMMs run on CTA pairs (256 x 256 tiles, M256 MMAs issued across two SMs);
WENC_GEMM_PAIR=0 keeps them on single CTAs (128 x 256 tiles, M128 MMAs). Either way each output
element is one dot product over K in the same order (16-element MMA steps, k-blocks in order), so
the outputs must agree bit for bit: for single GEMMs with every public epilogue, and for a
two-block forward at large-v3 dims, which also runs the LayerNorm-folded QKV and the statistics
epilogue of fc2. The single-CTA outputs are also held to the oracle, since no other test reaches
that form of the 256-column tiles."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import synth
from helpers import metrics

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _run_child(path, pair: bool):
    env = dict(os.environ)
    env["WENC_GEMM_PAIR"] = "1" if pair else "0"
    env["PYTHONPATH"] = os.pathsep.join([HERE, ROOT, env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, os.path.join(HERE, "gemm_forms_child.py"), str(path)], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return np.load(path)


def test_pair_and_single_cta_gemms_agree_bitwise(tmp_path):
    sys.path.insert(0, HERE)
    import gemm_forms_child as child
    single = _run_child(tmp_path / "single.npz", pair=False)
    pair = _run_child(tmp_path / "pair.npz", pair=True)
    assert sorted(single.files) == sorted(pair.files)
    for name in single.files:
        assert np.array_equal(single[name], pair[name]), name
    # the single-CTA outputs against the oracle (bf16 outputs: one rounding; f32: accumulation)
    for M, N, K, epi in child.LINEAR_CASES:
        rng = np.random.default_rng(1000 + M + N + K + epi)
        a = synth.round_to_bf16(rng.standard_normal((M, K)).astype(np.float32))
        wt = synth.round_to_bf16((0.05 * rng.standard_normal((N, K))).astype(np.float32))
        bias = (0.1 * rng.standard_normal(N)).astype(np.float32)
        resid = rng.standard_normal((M, N)).astype(np.float32) if epi == 2 else None
        z = oracle.linear(a, wt, bias)
        got = single[f"linear_{M}_{N}_{K}_{epi}"]
        if epi == 2:
            ref = resid.astype(np.float64) + z
            assert np.abs(got.astype(np.float64) - ref).max() <= 1e-4 * max(1.0, np.sqrt(np.mean(z * z)))
        else:
            ref = oracle.gelu(z) if epi == 1 else z
            got = synth.bf16_bits_to_f32(got.view(np.uint16)).astype(np.float64)
            assert (np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 2e-5 * np.sqrt(np.mean(ref * ref))).all(), \
                metrics(got, ref)
