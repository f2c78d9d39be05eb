"""Block and stack parity of wenc_forward / wenc_forward_layers against the f64 oracle.

Gates (the bf16 tensor-core bar): per block, max|err| <= 2e-2 x RMS and cosine >= 0.9999 on
the block output; the block's update y - x is gated too (2e-2 x RMS(y - x), cosine >= 0.999),
because the attention branch is small next to the residual and a wrong attention kernel
would otherwise hide under it. Per-block mode feeds block i the GPU's own output of block
i-1 (the bisection of turbospark-runtime encode_partial), so error does not compound.
Large stacks are checked on sampled rows of the first and last window: LN1, K and V run
over the whole window, the rest for the sampled rows only (exact for those rows).
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import gate, make_encoder

pytestmark = pytest.mark.gpu


def _t(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _block_gates(x_in, y_gpu, y_ref, what):
    gate(y_gpu, y_ref, what=f"{what} output")
    gate(y_gpu - x_in, y_ref - x_in, cos_min=0.999, what=f"{what} update")


def test_tiny_block_full():
    """One block, tiny dims, f32 weights (rounded to bf16 by the library), whole window."""
    import torch
    w = synth.WORKLOADS["tiny_block"]
    enc, layers, _, rng = make_encoder(w)
    x = synth.make_input(w, rng)
    y = enc.forward(_t(x))
    torch.cuda.synchronize()
    enc.sync_status()
    x1_ref, y_ref = oracle.encoder_block(x, layers[0], w.n_heads, return_mid=True)
    _block_gates(x.astype(np.float64), y.cpu().numpy(), y_ref, "tiny block")


def test_tiny_block_attention_branch_via_steps():
    """The attention half of the tiny block through the step entry points: x1 - x vs the oracle."""
    import torch
    from transformer_encoder_gb300 import attention, layernorm, linear
    w = synth.WORKLOADS["tiny_block"]
    _, layers, _, rng = make_encoder(w)
    p = layers[0]
    x = synth.make_input(w, rng)[0]
    d, H = w.d_model, w.n_heads
    xn = layernorm(_t(x), _t(p["ln1_w"]), _t(p["ln1_b"]))
    wqkv = _t(np.concatenate([p["wq"], p["wk"], p["wv"]])).to(torch.bfloat16)
    bqkv = _t(np.concatenate([p["bq"], np.zeros(d, np.float32), p["bv"]]))
    qkv = linear(xn, wqkv, bqkv, 0)
    q, k, v = (qkv[:, i * d:(i + 1) * d].contiguous().view(1, w.seq_len, H, 64) for i in range(3))
    o = attention(q, k, v).view(w.seq_len, d)
    x1 = linear(o, _t(p["wo"]).to(torch.bfloat16), _t(p["bo"]), 2, resid=_t(x))
    torch.cuda.synchronize()
    x1_ref, _ = oracle.encoder_block(x, p, H, return_mid=True)
    gate(x1.cpu().numpy() - x, x1_ref - x, cos_min=0.999, what="attention branch")


def _per_block(w, enc, layers, final, x, full: bool):
    """Run block by block on the GPU; compare each block (all rows or sampled rows)."""
    import torch
    cur = _t(x)
    B = w.batch
    sample = np.unique(np.r_[0, 1, 127, 128, 1407, 1408, w.seq_len - 1,
                             np.random.default_rng(0).integers(0, w.seq_len, 121)])
    for i, p in enumerate(layers):
        nxt = enc.forward_layers(cur, first=i, count=1, final_ln=False)
        torch.cuda.synchronize()
        x_in = cur.cpu().numpy().astype(np.float64)
        y = nxt.cpu().numpy()
        if full:
            y_ref = oracle.encoder_block(x_in, p, w.n_heads)
            _block_gates(x_in, y, y_ref, f"{w.name} block {i}")
        else:
            for b in sorted({0, B - 1}):
                _, y_ref = oracle.block_rows(x_in[b], sample, p, w.n_heads)
                _block_gates(x_in[b, sample], y[b, sample], y_ref, f"{w.name} block {i} window {b}")
        cur = nxt
    if final is not None:
        out = enc.forward_layers(cur, first=len(layers), count=0, final_ln=True)
        torch.cuda.synchronize()
        ref = oracle.layer_norm(cur.cpu().numpy(), final[0], final[1])
        gate(out.cpu().numpy(), ref, what=f"{w.name} final LN")
    return cur


def test_tiny_stack_per_block_and_whole():
    import torch
    w = synth.WORKLOADS["tiny_stack"]
    enc, layers, final, rng = make_encoder(w)
    x = synth.make_input(w, rng)
    last = _per_block(w, enc, layers, final, x, full=True)
    y = enc.forward(_t(x))
    torch.cuda.synchronize()
    # whole stack vs the oracle run end to end (errors compound over 4 blocks; same gate)
    gate(y.cpu().numpy(), oracle.encoder_stack(x, layers, w.n_heads, final=final), what="tiny stack end to end")
    # wenc_forward is exactly the per-block chain plus the final LN
    chained = enc.forward_layers(last, first=w.n_layers, count=0, final_ln=True)
    torch.cuda.synchronize()
    assert torch.equal(y, chained)


def test_base_stack_per_block_full():
    w = synth.WORKLOADS["base_stack"]
    enc, layers, final, rng = make_encoder(w)
    _per_block(w, enc, layers, final, synth.make_input(w, rng), full=True)


def test_small_stack_per_block_sampled():
    w = synth.WORKLOADS["small_stack"]
    enc, layers, final, rng = make_encoder(w)
    _per_block(w, enc, layers, final, synth.make_input(w, rng), full=False)


def test_large_stack_per_block_sampled():
    """Large-v3 dims, batch 16, 32 blocks: the launch configuration the bench times."""
    import torch
    w = synth.WORKLOADS["large_stack"]
    enc, layers, final, rng = make_encoder(w)
    x = synth.make_input(w, rng)
    last = _per_block(w, enc, layers, final, x, full=False)
    y = enc.forward(_t(x))
    chained = enc.forward_layers(last, first=w.n_layers, count=0, final_ln=True)
    torch.cuda.synchronize()
    assert torch.equal(y, chained)


def test_forward_in_place_and_partial_batch():
    import torch
    w = synth.WORKLOADS["tiny_stack"]
    enc, layers, final, rng = make_encoder(w, max_batch=3)
    x = np.concatenate([synth.make_input(w, rng, batch=3)])
    ref = enc.forward(_t(x))
    one = enc.forward(_t(x[1:2]))          # B < max_batch
    buf = _t(x)
    enc.forward(buf, out=buf)              # in place
    torch.cuda.synchronize()
    assert torch.equal(buf, ref)
    assert torch.equal(one[0], ref[1])     # windows are independent
    assert torch.equal(enc.forward(_t(x)), ref)  # deterministic


@pytest.mark.parametrize("precision", ["bf16", "tf32"])
def test_windows_independent_of_batch_large_dims(precision):
    """A window's output is the same bits whatever batch it runs in, at large-v3 dims (two blocks).

    The GEMMs cut a last partial wave into half-width units: at B = 1 every out-projection and fc2
    tile runs as two M128 N128 products, at B = 16 window 0's rows are whole 128 x 256 tiles; each
    output element must still be the same fixed-order dot product (no split of K, no batch-sized
    reduction)."""
    import torch
    w = synth.WORKLOADS["large_pair"]
    enc, _, _, rng = make_encoder(w, keep_host_layers=False, precision=precision)
    x = synth.make_input(w, rng)
    full = enc.forward(_t(x))
    first = enc.forward(_t(x[:1]))
    last = enc.forward(_t(x[-1:]))
    torch.cuda.synchronize()
    enc.sync_status()
    assert torch.equal(first[0], full[0])
    assert torch.equal(last[0], full[-1])


@pytest.mark.parametrize("wname,precision", [("tiny_stack", "bf16"), ("large_pair", "bf16"), ("large_pair", "tf32")])
def test_forward_captures_in_a_cuda_graph(wname, precision):
    """wenc_forward is stream-ordered and allocates nothing, so it can be captured into a CUDA
    graph (its launches keep their programmatic dependencies as graph edges); a replay gives the
    same bits as the eager call."""
    import torch
    w = synth.WORKLOADS[wname]
    enc, _, _, rng = make_encoder(w, keep_host_layers=False, precision=precision)
    x = _t(synth.make_input(w, rng))
    ref = enc.forward(x)
    out = torch.empty_like(x)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        enc.forward(x, out)  # a call on the capture stream before capturing
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        enc.forward(x, out)
    out.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    enc.sync_status()
    assert torch.equal(out, ref)


def test_concurrent_handles_from_two_host_threads():
    """Two host threads drive their own handles on their own streams at the same time (the
    binding releases the interpreter lock during library calls); every result equals the
    single-threaded one bit for bit, and the first calls of both threads race through the
    launchers' one-time set-up."""
    import threading
    import torch
    w = synth.WORKLOADS["tiny_stack"]
    encs, xs, refs = [], [], []
    for seed in (11, 12):
        enc, _, _, rng = make_encoder(w, keep_host_layers=False)
        x = _t(synth.make_input(w, np.random.default_rng(seed)))
        encs.append(enc)
        xs.append(x)
    outs = [[None] * 6 for _ in range(2)]
    errors = []

    def run(i):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for k in range(6):
                    outs[i][k] = encs[i].forward(xs[i])
            stream.synchronize()
        except Exception as e:  # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for i in range(2):
        encs[i].sync_status()
        ref = encs[i].forward(xs[i])
        torch.cuda.synchronize()
        for k in range(6):
            assert torch.equal(outs[i][k], ref)


def test_argument_errors():
    import torch
    from transformer_encoder_gb300 import WencError
    w = synth.WORKLOADS["tiny_block"]
    enc, _, _, rng = make_encoder(w)
    x = _t(synth.make_input(w, rng))
    with pytest.raises(WencError, match="INVALID_ARG"):
        enc.forward(torch.cat([x, x]))  # B = 2 > max_batch = 1
    with pytest.raises(WencError, match="INVALID_ARG"):
        enc.forward_layers(x, first=1, count=1)
    with pytest.raises(WencError, match="UNSUPPORTED"):
        from transformer_encoder_gb300 import attention
        q = torch.zeros(1, 8, 2, 32, dtype=torch.bfloat16, device="cuda")
        attention(q, q, q)
    enc.sync_status()


def test_split_key_attention_edge_shape():
    """T = 700 (six key tiles, the last with 60 keys), d = 128, one window: the handle splits the
    keys one tile per CTA and merges the partial results; the block must still match the oracle."""
    import torch
    from dataclasses import replace
    w = replace(synth.WORKLOADS["tiny_block"], name="split_edge", d_model=128, n_heads=2, ffn_dim=256, seq_len=700)
    enc, layers, _, rng = make_encoder(w)
    # row statistics, QKV (LN1 folded), attention, the split-key merge, out-proj, LN2, fc1, fc2
    assert enc.launches() == 8
    x = synth.make_input(w, rng)
    y = enc.forward(_t(x))
    torch.cuda.synchronize()
    enc.sync_status()
    y_ref = oracle.encoder_block(x, layers[0], w.n_heads)
    _block_gates(x.astype(np.float64), y.cpu().numpy(), y_ref, "split-key block")


def test_tiny_block_uses_split_keys():
    w = synth.WORKLOADS["tiny_block"]
    enc, _, _, _ = make_encoder(w)
    assert enc.launches() == 8  # 36 query-pair CTAs would fill a quarter of the GPU: keys are split
