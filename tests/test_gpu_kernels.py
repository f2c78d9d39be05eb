"""Step-level parity of the CUDA kernels (through the C ABI) against the f64 oracle.

Sizes span several tiles plus a ragged tail; inputs are seeded and synthetic.
Tolerances (derived from the arithmetic, stated per test):
  * bf16 outputs carry one rounding of at most 2^-9 relative; fp32 accumulation of bf16
    products adds ~1e-6 relative. So bf16 results are held to |err| <= 2^-8 |ref| + tiny.
  * fp32 outputs (LayerNorm f32, the residual epilogue) are held to 1e-5 of RMS / 2e-5 abs.
  * attention rounds P and its output to bf16: the elementwise bound of helpers.attention_gate
    (1.1 x 2^-9 (|o| + sum p|v|)), cosine >= 0.9999 and relative L2 error <= 1e-2.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import attention_gate, bf16_to_f64, gate, metrics

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    return torch


# ----------------------------------------------------------------------------- LayerNorm
@pytest.mark.parametrize("rows,d", [(1537, 384), (259, 512), (1500, 768), (1029, 1280), (1, 128)])
@pytest.mark.parametrize("out_bf16", [True, False])
def test_layernorm_matches_oracle(rows, d, out_bf16):
    torch = _torch()
    from transformer_encoder_gb300 import layernorm
    rng = np.random.default_rng(rows * 7 + d)
    x = (rng.standard_normal((rows, d)) * rng.uniform(0.1, 5, (rows, 1)) + rng.uniform(-3, 3, (rows, 1))).astype(np.float32)
    w = (1 + 0.02 * rng.standard_normal(d)).astype(np.float32)
    b = (0.02 * rng.standard_normal(d)).astype(np.float32)
    y = layernorm(torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(), torch.from_numpy(b).cuda(), 1e-5, out_bf16)
    torch.cuda.synchronize()
    ref = oracle.layer_norm(x, w, b, 1e-5)
    got = bf16_to_f64(y)
    if out_bf16:
        assert (np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6).all()
    else:
        assert np.abs(got - ref).max() <= 2e-5 * max(1.0, np.abs(ref).max())


# ----------------------------------------------------------------------------- GEMM + epilogues
# N % 256 == 0 runs on CTA pairs (256-row tiles): M = 1 and M = 100 leave the pair's second CTA
# without a valid row, M = 129 with one. M = 1500 and M = 24000 with N = 1280 run half-width
# units (all of them, or the last partial wave of a 470-tile launch).
@pytest.mark.parametrize("M,N,K", [(1537, 1152, 384), (300, 384, 1536), (1500, 2048, 512), (129, 256, 64),
                                   (3000, 1280, 1280), (6000, 1280, 512), (1537, 640, 256), (1, 256, 64),
                                   (100, 768, 192), (1500, 1280, 1280), (24000, 1280, 256)])
@pytest.mark.parametrize("epi", [0, 1, 2])
def test_linear_matches_oracle(M, N, K, epi):
    torch = _torch()
    from transformer_encoder_gb300 import linear
    rng = np.random.default_rng(M + N + K + epi)
    a = synth.round_to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    wt = synth.round_to_bf16((0.05 * rng.standard_normal((N, K))).astype(np.float32))
    bias = (0.1 * rng.standard_normal(N)).astype(np.float32)
    resid = rng.standard_normal((M, N)).astype(np.float32) if epi == 2 else None
    ta = torch.from_numpy(a).cuda().to(torch.bfloat16)
    tw = torch.from_numpy(wt).cuda().to(torch.bfloat16)
    tr = torch.from_numpy(resid).cuda() if resid is not None else None
    out = linear(ta, tw, torch.from_numpy(bias).cuda(), epi, resid=tr)
    torch.cuda.synchronize()
    z = oracle.linear(a, wt, bias)
    if epi == 0:
        ref = z
    elif epi == 1:
        ref = oracle.gelu(z)
    else:
        ref = resid.astype(np.float64) + z
    got = bf16_to_f64(out)
    if epi == 2:
        assert np.abs(got - ref).max() <= 1e-4 * max(1.0, np.sqrt(np.mean(z * z)))
    else:
        assert (np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 2e-5 * np.sqrt(np.mean(ref * ref))).all(), metrics(got, ref)


def test_linear_residual_in_place():
    torch = _torch()
    from transformer_encoder_gb300 import linear
    rng = np.random.default_rng(3)
    M, N, K = 700, 512, 256
    a = synth.round_to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    wt = synth.round_to_bf16((0.05 * rng.standard_normal((N, K))).astype(np.float32))
    bias = (0.1 * rng.standard_normal(N)).astype(np.float32)
    x = rng.standard_normal((M, N)).astype(np.float32)
    tx = torch.from_numpy(x).cuda()
    linear(torch.from_numpy(a).cuda().to(torch.bfloat16), torch.from_numpy(wt).cuda().to(torch.bfloat16),
           torch.from_numpy(bias).cuda(), 2, resid=tx, out=tx)
    torch.cuda.synchronize()
    ref = x + oracle.linear(a, wt, bias)
    assert np.abs(tx.cpu().numpy() - ref).max() <= 1e-4


# ----------------------------------------------------------------------------- attention
def _attn_case(B, T, H, scale, seed):
    torch = _torch()
    q, k, v = synth.make_qkv(B, T, H, 64, seed=seed, scale=scale)
    to_t = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    to_f = lambda a: synth.bf16_bits_to_f32(a).reshape(B, T, H * 64)
    return (to_t(q), to_t(k), to_t(v)), (to_f(q), to_f(k), to_f(v))


# T = 127 and 129 sit one key either side of the 128-key tile; T = 255 and 257 of two tiles (a
# query pair); B = 3 windows make the windows' rows interleave across work items.
@pytest.mark.parametrize("B,T,H", [(2, 1500, 3), (1, 256, 2), (3, 200, 1), (1, 64, 2), (1, 130, 1), (2, 3000, 1),
                                   (3, 127, 2), (1, 129, 2), (2, 255, 1), (1, 257, 3)])
@pytest.mark.parametrize("scale", [1.0, 0.1])
def test_attention_matches_oracle(B, T, H, scale):
    torch = _torch()
    from transformer_encoder_gb300 import attention
    (tq, tk, tv), (q, k, v) = _attn_case(B, T, H, scale, seed=1 + T)
    out = attention(tq, tk, tv)
    torch.cuda.synchronize()
    got = bf16_to_f64(out).reshape(B, T, H * 64)
    attention_gate(got, q, k, v, H, what=f"attention B={B} T={T} H={H} scale={scale}")


def test_attention_single_key_is_exact():
    # One key: p = 1, so out = v bit for bit.
    torch = _torch()
    from transformer_encoder_gb300 import attention
    (tq, tk, tv), _ = _attn_case(4, 1, 3, 1.0, seed=5)
    out = attention(tq, tk, tv)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), tv.view(torch.int16))


def test_attention_identical_keys_give_mean_value():
    torch = _torch()
    from transformer_encoder_gb300 import attention
    (tq, tk, tv), (q, k, v) = _attn_case(1, 777, 2, 1.0, seed=6)
    tk = tk[:, :1].expand_as(tk).contiguous()
    out = attention(tq, tk, tv)
    torch.cuda.synchronize()
    k = np.broadcast_to(k[:, :1], k.shape)
    ref = np.broadcast_to(v.astype(np.float64).mean(axis=1, keepdims=True), v.shape)
    got = bf16_to_f64(out).reshape(v.shape)
    attention_gate(got, q, k, v, 2, what="identical keys")
    # uniform p is exact in bf16, so only the fp32 sum and the output rounding remain
    assert (np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5).all()


def test_attention_sweep_shape_sampled_rows():
    """B=16, H=20 (large-v3 heads) at T in {256, 1500, 3000}: sampled query rows vs the oracle."""
    torch = _torch()
    from transformer_encoder_gb300 import attention
    B, H = 16, 20
    for T in (256, 1500, 3000):
        (tq, tk, tv), (q, k, v) = _attn_case(B, T, H, 1.0, seed=1)
        out = attention(tq, tk, tv)
        torch.cuda.synchronize()
        got = bf16_to_f64(out).reshape(B, T, H * 64)
        rows = np.unique(np.r_[0, 127, 128, T - 1, np.random.default_rng(T).integers(0, T, 60)])
        for b in (0, 7, B - 1):
            attention_gate(got[b, rows], q[b, rows], k[b], v[b], H, what=f"sweep T={T} b={b}")


def test_attention_deterministic():
    torch = _torch()
    from transformer_encoder_gb300 import attention
    (tq, tk, tv), _ = _attn_case(2, 1500, 4, 1.0, seed=9)
    o1 = attention(tq, tk, tv)
    o2 = attention(tq, tk, tv)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
