"""The decoder cross-attention K/V precompute (wenc_set_cross_kv / wenc_cross_kv) against the
f64 oracle.

One GEMM over all decoder layers writes K_l and V_l as planes [2 n_dec, B*T, d]. Bound, from
the arithmetic: the encoder output is rounded once to the operand format (u = 2^-9 for bf16,
2^-11 for TF32), the weights are exact on their grid (bf16 workloads) or rounded once (f32
weights), products accumulate in fp32 and the output is rounded once, so elementwise
|err| <= u (|ref| + w_r * sum_k |a_k||w_k|) with w_r = 1 (exact weights) or 2 (rounded weights);
the tests allow 1.1x that plus 1e-6, and a relative L2 error of at most 2u.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import make_encoder

pytestmark = pytest.mark.gpu


def _t(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _attach(enc, w, n_dec=None):
    import torch
    dec = synth.make_cross(w, n_dec)
    dev = []
    for p in dec:
        q = {k: _t(v) for k, v in p.items()}
        if w.bf16_weights:
            q["wk"], q["wv"] = q["wk"].to(torch.bfloat16), q["wv"].to(torch.bfloat16)
        dev.append(q)
    enc.set_cross_kv(dev)
    return dec


def _check(got, enc_out, dec, rows, precision, weights_exact, what):
    """got: [2L, len(rows), d] float64; rows index the flattened [B*T] positions."""
    u = 2.0 ** -11 if precision == "tf32" else 2.0 ** -9
    wr = 1.0 if weights_exact else 2.0
    a = enc_out.reshape(-1, enc_out.shape[-1])[rows].astype(np.float64)
    ref = oracle.cross_kv(a, [p["wk"] for p in dec], [p["wv"] for p in dec], [p["bv"] for p in dec])
    for l, p in enumerate(dec):
        for j, key in enumerate(("wk", "wv")):
            plane = 2 * l + j
            absz = np.abs(a) @ np.abs(p[key].astype(np.float64)).T
            bound = 1.1 * u * (np.abs(ref[plane]) + wr * absz) + 1e-6
            err = np.abs(got[plane] - ref[plane])
            assert (err <= bound).all(), f"{what} plane {plane}: {float((err / bound).max()):.2f} x the bound"
    rel_l2 = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert rel_l2 <= 2 * u, f"{what}: relative L2 error {rel_l2:.3e}"


def _to_f64(t):
    import torch
    return t.to(torch.float32).cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("precision", ["bf16", "tf32"])
def test_cross_kv_tiny_dims(precision):
    """d = 384, four decoder layers, two windows; every output checked."""
    import torch
    w = synth.WORKLOADS["tiny_stack"]
    enc, _, _, _ = make_encoder(w, keep_host_layers=False, max_batch=2, precision=precision)
    dec = _attach(enc, w)
    enc_out = np.random.default_rng(21).standard_normal((2, w.seq_len, w.d_model)).astype(np.float32)
    kv = enc.cross_kv(_t(enc_out))
    torch.cuda.synchronize()
    enc.sync_status()
    assert tuple(kv.shape) == (2 * w.n_layers, 2 * w.seq_len, w.d_model)
    _check(_to_f64(kv), enc_out, dec, np.arange(2 * w.seq_len), precision, True, f"{precision} cross K/V tiny")


def test_cross_kv_f32_weights_and_partial_batch():
    """f32 decoder weights (rounded by the library) and a call with B below max_batch."""
    import torch
    w = synth.WORKLOADS["tiny_block"]
    enc, _, _, _ = make_encoder(w, keep_host_layers=False, max_batch=3)
    dec = _attach(enc, w, n_dec=2)
    enc_out = np.random.default_rng(22).standard_normal((1, w.seq_len, w.d_model)).astype(np.float32)
    kv = enc.cross_kv(_t(enc_out))
    torch.cuda.synchronize()
    enc.sync_status()
    assert tuple(kv.shape) == (4, w.seq_len, w.d_model)
    _check(_to_f64(kv), enc_out, dec, np.arange(w.seq_len), "bf16", False, "cross K/V f32 weights")


def test_cross_kv_large_dims_sampled_rows():
    """Large-v3 dims: 32 decoder layers (N = 81920), 16 windows; 64 sampled rows of every plane."""
    import torch
    w = synth.WORKLOADS["large_stack"]
    enc, _, _, _ = make_encoder(w, keep_host_layers=False)
    dec = _attach(enc, w)
    enc_out = np.random.default_rng(23).standard_normal((w.batch, w.seq_len, w.d_model)).astype(np.float32)
    kv = enc.cross_kv(_t(enc_out))
    torch.cuda.synchronize()
    enc.sync_status()
    M = w.batch * w.seq_len
    rows = np.unique(np.r_[0, 1, 127, 128, 1499, 1500, M - 1, np.random.default_rng(0).integers(0, M, 57)])
    got = _to_f64(kv[:, torch.from_numpy(rows).cuda()])
    _check(got, enc_out, dec, rows, "bf16", True, "cross K/V large")


def test_cross_kv_after_encode_and_errors():
    """On the encoder's own output, and the argument checks."""
    import torch
    from transformer_encoder_gb300 import WencError
    w = synth.WORKLOADS["tiny_stack"]
    enc, _, _, rng = make_encoder(w, keep_host_layers=False)
    x = _t(synth.make_input(w, rng))
    with pytest.raises(WencError, match="cross"):
        enc.cross_kv(x)  # no weights attached yet
    dec = _attach(enc, w)
    y = enc.forward(x)
    kv = enc.cross_kv(y)
    torch.cuda.synchronize()
    enc.sync_status()
    _check(_to_f64(kv), y.cpu().numpy(), dec, np.arange(w.seq_len), "bf16", True, "cross K/V of the encoder output")
