"""The TF32 precision (WENC_PREC_TF32) against the f64 oracle.

Every contraction runs on the tensor cores with TF32 operands (10 explicit mantissa bits,
rounded to nearest by the kernel that writes them) and fp32 accumulation; activations between
kernels are fp32. Gates:
  * blocks and stacks: max|err| <= 1e-3 x RMS of the output and cosine >= 0.99999 (the
    "1e-3 relative" bar for the TF32/FP32 path); the block's update y - x (the part the block
    computes, small next to the residual) within 5e-3 x its RMS and a relative L2 error
    <= 1.5e-3. A CPU model of the same roundings gives 3.7e-4, 2.2e-3 and 4.2e-4 on the tiny
    block (4.9e-4 end to end over the tiny stack); the bf16 path gives 2.6e-3, 1.6e-2 and
    3.3e-3, so the gates tell the two precisions apart.
  * kernels: one TF32 rounding (<= 2^-11 relative) of each written operand plus fp32
    accumulation, as stated per test.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import attention_gate, gate, make_encoder, metrics

pytestmark = pytest.mark.gpu

U = 2.0 ** -11  # TF32 unit roundoff (round to nearest)


def _t(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _on_tf32_grid(t) -> bool:
    import torch
    bits = t.contiguous().view(torch.int32)
    return bool(((bits & 0x1FFF) == 0).all().item())


# ----------------------------------------------------------------------------- LayerNorm
@pytest.mark.parametrize("rows,d", [(1537, 384), (259, 512), (1029, 1280), (1, 128)])
def test_layernorm_tf32_output(rows, d):
    import torch
    from transformer_encoder_gb300 import LN_OUT_TF32, layernorm
    rng = np.random.default_rng(rows * 5 + d)
    x = (rng.standard_normal((rows, d)) * rng.uniform(0.1, 5, (rows, 1)) + rng.uniform(-3, 3, (rows, 1))).astype(np.float32)
    w = (1 + 0.02 * rng.standard_normal(d)).astype(np.float32)
    b = (0.02 * rng.standard_normal(d)).astype(np.float32)
    y = layernorm(_t(x), _t(w), _t(b), 1e-5, out_format=LN_OUT_TF32)
    torch.cuda.synchronize()
    assert y.dtype == torch.float32 and _on_tf32_grid(y)
    ref = oracle.layer_norm(x, w, b, 1e-5)
    got = y.cpu().numpy().astype(np.float64)
    # one TF32 rounding of the fp32 result, whose own error is held to 2e-5 of max|ref|
    assert (np.abs(got - ref) <= 1.001 * U * np.abs(ref) + 2e-5 * max(1.0, np.abs(ref).max())).all()


# ----------------------------------------------------------------------------- GEMM + epilogues
@pytest.mark.parametrize("M,N,K", [(1537, 1152, 384), (300, 384, 1536), (129, 256, 96), (1500, 128, 32),
                                   (3000, 1280, 1280), (1537, 640, 256)])
@pytest.mark.parametrize("epi", [0, 1, 2])
def test_linear_tf32_matches_oracle(M, N, K, epi):
    """Operands on the TF32 grid; the product is exact in fp32, accumulation adds at most
    2^-16 of sum |a||w| here; epilogues 0 and 1 add one TF32 rounding of the output."""
    import torch
    from transformer_encoder_gb300 import linear_tf32, sync_status
    rng = np.random.default_rng(M + N + K + 10 * epi)
    a = synth.round_to_tf32(rng.standard_normal((M, K)).astype(np.float32))
    wt = synth.round_to_tf32((0.05 * rng.standard_normal((N, K))).astype(np.float32))
    bias = (0.1 * rng.standard_normal(N)).astype(np.float32)
    resid = rng.standard_normal((M, N)).astype(np.float32) if epi == 2 else None
    out = linear_tf32(_t(a), _t(wt), _t(bias), epi, resid=_t(resid) if resid is not None else None)
    torch.cuda.synchronize()
    sync_status()
    z = oracle.linear(a, wt, bias)
    absz = np.abs(a.astype(np.float64)) @ np.abs(wt.astype(np.float64)).T
    acc = 2.0 ** -16 * absz + 1e-6
    if epi == 0:
        ref = z
    elif epi == 1:
        ref = oracle.gelu(z)
    else:
        ref = resid.astype(np.float64) + z
    got = out.cpu().numpy().astype(np.float64)
    if epi == 2:
        assert (np.abs(got - ref) <= acc + 2.0 ** -23 * np.abs(ref)).all(), metrics(got, ref)
    else:
        assert _on_tf32_grid(out)
        assert (np.abs(got - ref) <= 1.001 * U * np.abs(ref) + acc).all(), metrics(got, ref)
        # a bf16 reading of the operands would leave about 2^-9 relative error
        rel_l2 = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel_l2 <= U, rel_l2


# ----------------------------------------------------------------------------- attention
def _attn_case(B, T, H, scale, seed):
    rng = np.random.default_rng(seed)
    arrs = [synth.round_to_tf32((scale * rng.standard_normal((B, T, H, 64))).astype(np.float32)) for _ in range(3)]
    return [_t(a) for a in arrs], [a.reshape(B, T, H * 64) for a in arrs]


@pytest.mark.parametrize("B,T,H", [(2, 1500, 3), (1, 256, 2), (3, 200, 1), (1, 64, 2), (1, 65, 1), (1, 130, 1),
                                   (2, 3000, 1)])
@pytest.mark.parametrize("scale", [1.0, 0.1])
def test_attention_tf32_matches_oracle(B, T, H, scale):
    import torch
    from transformer_encoder_gb300 import attention_tf32, sync_status
    (tq, tk, tv), (q, k, v) = _attn_case(B, T, H, scale, seed=3 + T + H)
    out = attention_tf32(tq, tk, tv)
    torch.cuda.synchronize()
    sync_status()  # no bounded wait of the kernel ran out
    assert _on_tf32_grid(out)
    got = out.cpu().numpy().astype(np.float64).reshape(B, T, H * 64)
    attention_gate(got, q, k, v, H, what=f"TF32 attention B={B} T={T} H={H} scale={scale}", tf32=True)


def test_attention_tf32_single_key_is_exact():
    # One key: p = 1, so out = v bit for bit (v is on the TF32 grid).
    import torch
    from transformer_encoder_gb300 import attention_tf32
    (tq, tk, tv), _ = _attn_case(4, 1, 3, 1.0, seed=5)
    out = attention_tf32(tq, tk, tv)
    torch.cuda.synchronize()
    assert torch.equal(out, tv)


def test_attention_tf32_identical_keys_give_mean_value():
    import torch
    from transformer_encoder_gb300 import attention_tf32
    (tq, tk, tv), (q, k, v) = _attn_case(1, 777, 2, 1.0, seed=6)
    tk = tk[:, :1].expand_as(tk).contiguous()
    out = attention_tf32(tq, tk, tv)
    torch.cuda.synchronize()
    k = np.broadcast_to(k[:, :1], k.shape)
    ref = np.broadcast_to(v.astype(np.float64).mean(axis=1, keepdims=True), v.shape)
    got = out.cpu().numpy().astype(np.float64).reshape(v.shape)
    attention_gate(got, q, k, v, 2, what="TF32 identical keys", tf32=True)
    # every probability is exactly 1: only the fp32 sum and the output rounding remain
    assert (np.abs(got - ref) <= 1.001 * U * np.abs(ref) + 1e-5).all()


# ----------------------------------------------------------------------------- blocks and stacks
def _tf32_block_gates(x_in, y_gpu, y_ref, what):
    gate(y_gpu, y_ref, rel=1e-3, cos_min=0.99999, what=f"{what} output")
    upd, upd_ref = y_gpu - x_in, y_ref - x_in
    gate(upd, upd_ref, rel=5e-3, cos_min=0.99999, what=f"{what} update")
    rel_l2 = float(np.linalg.norm(upd - upd_ref) / np.linalg.norm(upd_ref))
    assert rel_l2 <= 1.5e-3, f"{what}: update relative L2 error {rel_l2:.3e}"


def test_tf32_tiny_block_full():
    """One block, tiny dims, the f32 weights as given (rounded to TF32 by the library)."""
    import torch
    w = synth.WORKLOADS["tiny_block"]
    enc, layers, _, rng = make_encoder(w, precision="tf32")
    x = synth.make_input(w, rng)
    y = enc.forward(_t(x))
    torch.cuda.synchronize()
    enc.sync_status()
    y_ref = oracle.encoder_block(x, layers[0], w.n_heads)
    _tf32_block_gates(x.astype(np.float64), y.cpu().numpy(), y_ref, "TF32 tiny block")


def test_tf32_tiny_stack_per_block_and_whole():
    import torch
    w = synth.WORKLOADS["tiny_stack"]
    enc, layers, final, rng = make_encoder(w, precision="tf32")
    x = synth.make_input(w, rng)
    cur = _t(x)
    for i, p in enumerate(layers):
        nxt = enc.forward_layers(cur, first=i, count=1, final_ln=False)
        torch.cuda.synchronize()
        x_in = cur.cpu().numpy().astype(np.float64)
        _tf32_block_gates(x_in, nxt.cpu().numpy(), oracle.encoder_block(x_in, p, w.n_heads), f"TF32 tiny block {i}")
        cur = nxt
    y = enc.forward(_t(x))
    torch.cuda.synchronize()
    enc.sync_status()
    ref = oracle.encoder_stack(x, layers, w.n_heads, final=final)
    gate(y.cpu().numpy(), ref, rel=1e-3, cos_min=0.99999, what="TF32 tiny stack end to end")
    chained = enc.forward_layers(cur, first=w.n_layers, count=0, final_ln=True)
    torch.cuda.synchronize()
    assert torch.equal(y, chained)


def test_tf32_ragged_window_two_batches():
    """700-frame windows (a partial 128-query tile and a partial 64-key tile), two windows in
    one call, tiny dims: attention must not mix windows or read past a window's end."""
    import torch
    w = synth.WORKLOADS["tiny_block"]
    enc, layers, _, rng = make_encoder(w, precision="tf32", seq_len=700, max_batch=2)
    x = rng.standard_normal((2, 700, w.d_model), dtype=np.float32)
    y = enc.forward(_t(x))
    torch.cuda.synchronize()
    enc.sync_status()
    y_ref = oracle.encoder_block(x, layers[0], w.n_heads)
    _tf32_block_gates(x.astype(np.float64), y.cpu().numpy(), y_ref, "TF32 T=700 B=2 block")


def test_tf32_and_bf16_handles_launch_the_same_sequence():
    import torch
    w = synth.WORKLOADS["tiny_stack"]
    enc, _, _, _ = make_encoder(w, keep_host_layers=False, precision="tf32")
    assert enc.precision == "tf32"
    # LN, QKV, attention (one kernel: no key split), out-proj, LN, fc1, fc2 per block + final LN
    assert enc.launches() == 7 * w.n_layers + 1
    events = [torch.cuda.Event(enable_timing=True) for _ in range(enc.launches() + 1)]
    for e in events:
        e.record()
    kinds = enc.set_launch_events(events)
    x = _t(synth.make_input(w, np.random.default_rng(0)))
    enc.forward(x)
    torch.cuda.synchronize()
    assert list(kinds)[:7] == [0, 1, 2, 3, 0, 4, 5] and kinds[7 * w.n_layers] == 6
