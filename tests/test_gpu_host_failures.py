"""Failures made on the host, with no GPU fault: device allocations that run out (through the
library's allocation cap) and a stream that is being captured into a CUDA graph.

The pages' error contract is a status returned to the caller, never an abort: turbospark-runtime
encode_partial rejects a wrong frame count with an error, oxinfer WhisperConfig validates its
dimensions before any work. Here wenc_create, wenc_set_stem and wenc_set_cross_kv must return
WENC_ERR_OOM when an allocation fails and keep nothing allocated, and refuse a capturing stream
before touching it.
"""
import ctypes

import numpy as np
import pytest

import synth
from helpers import make_encoder, upload_layer

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS["tiny_stack"]


def _layers():
    import torch
    layers, final, rng = synth.make_weights(W)
    dev = [upload_layer(p, W.bf16_weights) for p in layers]
    fin = (torch.from_numpy(final[0]).cuda(), torch.from_numpy(final[1]).cuda())
    return dev, fin, rng


def _stem(enc_dtype):
    import torch
    st = synth.make_stem(W)
    return {k: (torch.from_numpy(v).to(enc_dtype) if k in ("conv1_w", "conv2_w") else torch.from_numpy(v)).cuda()
            for k, v in st.items()}


def _cross(enc_dtype, n=2):
    import torch
    return [{"wk": torch.from_numpy(p["wk"]).to(enc_dtype).cuda(), "wv": torch.from_numpy(p["wv"]).to(enc_dtype).cuda(),
             "bv": torch.from_numpy(p["bv"]).cuda()} for p in synth.make_cross(W, n)]


@pytest.fixture
def lib_cap():
    from transformer_encoder_gb300 import lib
    L = lib()
    yield L
    L.wenc_set_device_alloc_limit(0)


def test_create_out_of_memory_keeps_nothing(lib_cap):
    import torch
    from transformer_encoder_gb300 import Encoder, WencError
    L = lib_cap
    dev, fin, rng = _layers()
    held0 = L.wenc_device_bytes_held()
    enc = Encoder(dev, W.n_heads, W.seq_len, W.batch, final=fin)
    need = L.wenc_device_bytes_held() - held0  # weights + workspace of one handle
    assert need > 0
    x = torch.from_numpy(synth.make_input(W, rng)).cuda()
    ref = enc.forward(x)
    torch.cuda.synchronize()
    enc.close()
    assert L.wenc_device_bytes_held() == held0
    # a cap that stops the first allocation (weights), then one that stops the second (workspace)
    for cap, what in ((1, "weights"), (need - 1, "workspace")):
        L.wenc_set_device_alloc_limit(held0 + cap)
        with pytest.raises(WencError, match="OOM") as ei:
            Encoder(dev, W.n_heads, W.seq_len, W.batch, final=fin)
        assert what in str(ei.value)
        assert L.wenc_device_bytes_held() == held0
    L.wenc_set_device_alloc_limit(0)
    enc = Encoder(dev, W.n_heads, W.seq_len, W.batch, final=fin)
    got = enc.forward(x)
    torch.cuda.synchronize()
    enc.sync_status()
    assert torch.equal(got, ref)
    enc.close()
    assert L.wenc_device_bytes_held() == held0


def test_set_stem_and_cross_kv_out_of_memory_leave_the_handle_working(lib_cap):
    import torch
    from transformer_encoder_gb300 import WencError
    L = lib_cap
    enc, _, _, rng = make_encoder(W, keep_host_layers=False)
    x = torch.from_numpy(synth.make_input(W, rng)).cuda()
    ref = enc.forward(x)
    torch.cuda.synchronize()
    held = L.wenc_device_bytes_held()
    L.wenc_set_device_alloc_limit(held)  # no room for anything more
    with pytest.raises(WencError, match="OOM") as ei:
        enc.set_stem(_stem(torch.bfloat16))
    assert "stem" in str(ei.value)
    assert L.wenc_device_bytes_held() == held
    with pytest.raises(WencError, match="OOM") as ei:
        enc.set_cross_kv(_cross(torch.bfloat16))
    assert "cross" in str(ei.value)
    assert L.wenc_device_bytes_held() == held
    got = enc.forward(x)  # the handle still computes, bit-equal to before
    torch.cuda.synchronize()
    enc.sync_status()
    assert torch.equal(got, ref)
    with pytest.raises(WencError, match="INVALID_ARG"):  # no stem was attached
        enc.encode(torch.zeros((W.batch, 2 * W.seq_len, W.n_mels), device="cuda"))
    L.wenc_set_device_alloc_limit(0)
    enc.set_stem(_stem(torch.bfloat16))
    enc.set_cross_kv(_cross(torch.bfloat16))
    assert L.wenc_device_bytes_held() > held
    enc.close()


def test_capturing_stream_is_refused_and_the_capture_survives():
    import torch
    from transformer_encoder_gb300 import Encoder, WencError, lib
    L = lib()
    dev, fin, rng = _layers()
    enc = Encoder(dev, W.n_heads, W.seq_len, W.batch, final=fin)
    x = torch.from_numpy(synth.make_input(W, rng)).cuda()
    out = torch.empty_like(x)
    enc.forward(x, out)
    torch.cuda.synchronize()
    ref = out.clone()
    stem = _stem(torch.bfloat16)  # made before the capture: its host-to-device copies are not capturable
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    errors = []
    with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
        try:
            Encoder(dev, W.n_heads, W.seq_len, W.batch, final=fin, stream=s)
        except WencError as e:
            errors.append(("create", str(e)))
        try:
            enc.set_stem(stem, stream=s)
        except WencError as e:
            errors.append(("set_stem", str(e)))
        enc.forward(x, out, stream=s)  # forward is stream-ordered: it is captured
    assert [w for w, _ in errors] == ["create", "set_stem"]
    assert all("INVALID_ARG" in m and "captured" in m for _, m in errors)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    enc.sync_status()
    assert torch.equal(out, ref)
    enc.close()
