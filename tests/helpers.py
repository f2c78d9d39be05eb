"""Shared helpers of the parity tests: uploads, gates and comparisons (no encoder arithmetic)."""
from __future__ import annotations

import numpy as np

import synth


def metrics(gpu, ref):
    """max|err|, RMS(ref), cosine between two arrays (float64)."""
    g = np.asarray(gpu, np.float64).ravel()
    r = np.asarray(ref, np.float64).ravel()
    err = np.abs(g - r).max() if g.size else 0.0
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    den = np.linalg.norm(g) * np.linalg.norm(r)
    cos = float(g @ r / den) if den > 0 else 1.0
    return float(err), rms, cos


def gate(gpu, ref, rel=2e-2, cos_min=0.9999, what=""):
    """The bf16 tensor-core gate: max|err| <= rel * RMS(ref) and cosine >= cos_min."""
    err, rms, cos = metrics(gpu, ref)
    assert np.isfinite(np.asarray(gpu, np.float64)).all(), f"{what}: non-finite output"
    assert err <= rel * rms, f"{what}: max|err| {err:.3e} > {rel} * RMS {rms:.3e} (cos {cos:.6f})"
    assert cos >= cos_min, f"{what}: cosine {cos:.6f} < {cos_min} (max|err| {err:.3e}, RMS {rms:.3e})"
    return err, rms, cos


def attention_gate(got, q, k, v, n_heads, what="", tf32=False):
    """Gate for an attention output, derived from its arithmetic.

    bf16 kernel: each probability p_j is rounded to bf16 before the PV product and the output
    is rounded to bf16; everything else is fp32 (relative error ~1e-6). Each rounding is at
    most u = 2^-9 relative, so |o_gpu - o| <= u (|o| + sum_j p_j |v_j|) elementwise.
    TF32 kernel: u = 2^-11 (TF32 keeps 10 explicit mantissa bits, rounded to nearest), and
    the denominator is the sum of the rounded probabilities, whose own relative deviation
    (<= u) adds u |o|: |o_gpu - o| <= u (2 |o| + sum_j p_j |v_j|).
    The test allows 1.1x that worst case (fp32 accumulation of up to a few thousand terms),
    plus a cosine >= 0.9999 and a relative L2 error <= 1e-2 (bf16) or 2e-3 (TF32), which
    catch systematic mistakes that stay under the elementwise bound (a dropped or
    sign-flipped key, a wrong mask).
    """
    import oracle
    ref = oracle.attention(q, k, v, n_heads)
    absv = oracle.attention(q, k, np.abs(np.asarray(v, np.float64)), n_heads)
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    u, n_o, l2_max = (2.0 ** -11, 2.0, 2e-3) if tf32 else (2.0 ** -9, 1.0, 1e-2)
    bound = 1.1 * u * (n_o * np.abs(ref) + absv) + 1e-6
    worst = float((err / bound).max())
    _, rms, cos = metrics(got, ref)
    rel_l2 = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    kind = "TF32" if tf32 else "bf16"
    assert worst <= 1.0, f"{what}: error reaches {worst:.2f} x the {kind} rounding bound (max|err| {err.max():.3e})"
    assert cos >= 0.9999, f"{what}: cosine {cos:.6f}"
    assert rel_l2 <= l2_max, f"{what}: relative L2 error {rel_l2:.3e}"
    return worst, cos, rel_l2


def bf16_to_f64(t):
    """A torch bf16 tensor (GPU or CPU) as a float64 numpy array."""
    import torch
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def upload_layer(p: dict, bf16_matrices: bool, device="cuda"):
    """Host float32 parameter dict -> CUDA tensors (matrices bf16 or f32, vectors f32)."""
    import torch
    out = {}
    for k, v in p.items():
        t = torch.from_numpy(np.ascontiguousarray(v))
        if k in synth.MATRIX_KEYS and bf16_matrices:
            t = t.to(torch.bfloat16)  # exact: the values are already bf16-representable
        out[k] = t.to(device)
    return out


def make_encoder(w: synth.Workload, keep_host_layers: bool = True, max_batch: int | None = None,
                 precision: str = "bf16", seq_len: int | None = None):
    """Draw a workload's parameters, build the GPU encoder from them, return (enc, layers, final, rng)."""
    import torch
    from transformer_encoder_gb300 import Encoder

    host_layers = []
    dev_layers = []

    def cb(p):
        dev_layers.append(upload_layer(p, w.bf16_weights))
        if keep_host_layers:
            host_layers.append(p)
        return None

    _, final, rng = synth.make_weights(w, layer_callback=cb)
    fin_dev = (torch.from_numpy(final[0]).cuda(), torch.from_numpy(final[1]).cuda()) if w.final_ln else None
    enc = Encoder(dev_layers, w.n_heads, seq_len or w.seq_len, max_batch or w.batch, final=fin_dev,
                  precision=precision)
    del dev_layers
    torch.cuda.synchronize()
    return enc, host_layers, final, rng
