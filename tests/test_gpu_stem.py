"""The convolutional stem (wenc_set_stem / wenc_stem / wenc_encode) against the f64 oracle.

The stem's output is GELU(conv2) + positions; the positional rows (exact copies) dominate its
RMS, so the convolution part y - positions is gated on its own as well. Gates, from a CPU model
of the path's roundings (operands rounded to bf16 or TF32 where the kernels round them):
  * bf16: output max|err| <= 2e-2 x RMS, cosine >= 0.9999; conv part max|err| <= 4e-2 x its
    RMS, relative L2 <= 1e-2 (model: 1.6e-2 and 3.2e-3 on the tiny dims, 1.5e-2 and 2.3e-3 at
    large-v3 dims);
  * TF32: output max|err| <= 1e-3 x RMS; conv part max|err| <= 5e-3 x RMS, relative L2 <= 1.5e-3
    (model: 2.2e-3 and 4.0e-4).
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import gate, make_encoder

pytestmark = pytest.mark.gpu

GATES = {"bf16": dict(out=2e-2, cos=0.9999, conv=4e-2, l2=1e-2),
         "tf32": dict(out=1e-3, cos=0.99999, conv=5e-3, l2=1.5e-3)}


def _t(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _attach_stem(enc, w):
    import torch
    p = synth.make_stem(w)
    dev = {}
    for k, v in p.items():
        t = _t(v)
        if k in ("conv1_w", "conv2_w") and w.bf16_weights:
            t = t.to(torch.bfloat16)  # exact: drawn on the bf16 grid
        dev[k] = t
    enc.set_stem(dev)
    return p


def _stem_ref(mel, p):
    return oracle.conv_stem(mel, p["conv1_w"], p["conv1_b"], p["conv2_w"], p["conv2_b"], p["positions"])


def _stem_gates(got, ref, pos, precision, what):
    g = GATES[precision]
    gate(got, ref, rel=g["out"], cos_min=g["cos"], what=f"{what} output")
    conv, conv_ref = got - pos, ref - pos
    gate(conv, conv_ref, rel=g["conv"], cos_min=0.999, what=f"{what} conv part")
    rel_l2 = float(np.linalg.norm(conv - conv_ref) / np.linalg.norm(conv_ref))
    assert rel_l2 <= g["l2"], f"{what}: conv part relative L2 error {rel_l2:.3e}"


@pytest.mark.parametrize("precision", ["bf16", "tf32"])
def test_stem_tiny_dims(precision):
    """Tiny dims (80 mel bands, d = 384), two windows, f32 weights."""
    import torch
    w = synth.WORKLOADS["tiny_block"]
    enc, _, _, _ = make_encoder(w, keep_host_layers=False, max_batch=2, precision=precision)
    p = _attach_stem(enc, w)
    mel = synth.make_mel(w, batch=2)
    x = enc.stem(_t(mel))
    torch.cuda.synchronize()
    enc.sync_status()
    ref = _stem_ref(mel, p)
    _stem_gates(x.cpu().numpy(), ref, p["positions"], precision, f"{precision} stem tiny")


def test_stem_ragged_window_length():
    """700-position windows (1400 mel frames): partial GEMM tiles and a positional period of 700."""
    import torch
    w = synth.WORKLOADS["tiny_block"]
    T = 700
    enc, _, _, _ = make_encoder(w, keep_host_layers=False, max_batch=2, seq_len=T)
    p = synth.make_stem(w)
    p["positions"] = np.ascontiguousarray(p["positions"][:T])
    enc.set_stem({k: _t(v) for k, v in p.items()})
    mel = np.random.default_rng(3).uniform(-1, 1, (2, 2 * T, w.n_mels)).astype(np.float32)
    x = enc.stem(_t(mel))
    torch.cuda.synchronize()
    enc.sync_status()
    _stem_gates(x.cpu().numpy(), _stem_ref(mel, p), p["positions"], "bf16", "stem T=700")


def test_stem_large_dims_first_and_last_window():
    """Large-v3 dims (128 mel bands, d = 1280) at batch 16, bf16 weights: windows 0 and 15."""
    import torch
    w = synth.WORKLOADS["large_block"]
    enc, _, _, _ = make_encoder(w, keep_host_layers=False)
    p = _attach_stem(enc, w)
    mel = synth.make_mel(w)
    x = enc.stem(_t(mel))
    torch.cuda.synchronize()
    enc.sync_status()
    got = x.cpu().numpy()
    for b in (0, w.batch - 1):
        _stem_gates(got[b], _stem_ref(mel[b], p), p["positions"], "bf16", f"large stem window {b}")


@pytest.mark.parametrize("precision", ["bf16", "tf32"])
def test_encode_is_stem_then_blocks(precision):
    """wenc_encode = the stem, every block and the final LN: against the oracle end to end, and bit
    for bit against wenc_stem followed by wenc_forward."""
    import torch
    w = synth.WORKLOADS["tiny_stack"]
    enc, layers, final, _ = make_encoder(w, precision=precision)
    p = _attach_stem(enc, w)
    mel = synth.make_mel(w, batch=1)
    y = enc.encode(_t(mel))
    chained = enc.forward(enc.stem(_t(mel)))
    torch.cuda.synchronize()
    enc.sync_status()
    assert torch.equal(y, chained)
    ref = oracle.encoder_stack(_stem_ref(mel, p), layers, w.n_heads, final=final)
    g = GATES[precision]
    gate(y.cpu().numpy(), ref, rel=g["out"], cos_min=g["cos"], what=f"{precision} encode from mel")


def test_encode_launch_accounting_and_errors():
    import torch
    from transformer_encoder_gb300 import WencError
    w = synth.WORKLOADS["tiny_stack"]
    enc, _, _, _ = make_encoder(w, keep_host_layers=False)
    mel = _t(synth.make_mel(w, batch=1))
    with pytest.raises(WencError, match="stem"):
        enc.encode(mel)  # no stem attached yet
    assert enc.encode_launches() == -1
    _attach_stem(enc, w)
    n = enc.encode_launches()
    assert n == 4 + enc.launches()
    events = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    for e in events:
        e.record()
    kinds = enc.set_launch_events(events)
    enc.encode(mel)
    torch.cuda.synchronize()
    assert list(kinds)[:5] == [9, 10, 9, 11, 14]  # the stem, then the blocks' row statistics
    with pytest.raises(WencError):
        enc.encode(_t(synth.make_mel(w, batch=2)))  # B above max_batch
