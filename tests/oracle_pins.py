"""Pins that tie the f64 oracle to facts fixed outside itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with a
hand-worked fixture (tests/golden/, each with its source), a closed form, an
invariant, or PyTorch's float64 CPU modules on a special case that reduces to
them. The functions look the oracle up through ``oracle.encoder`` at call time,
so ``test_oracle_mutations.py`` can plant mistakes in it and check that some
pin catches each one.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle.encoder as E
import oracle.stem as S
import oracle.cross as X

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _close(a, b, rtol=1e-12, atol=1e-12):
    np.testing.assert_allclose(np.asarray(a, np.float64), np.asarray(b, np.float64), rtol=rtol, atol=atol)


def _rand_params(rng, d, f, scale=0.3):
    n = lambda *s: rng.standard_normal(s) * scale
    return {
        "ln1_w": 1 + n(d), "ln1_b": n(d), "wq": n(d, d), "bq": n(d), "wk": n(d, d),
        "wv": n(d, d), "bv": n(d), "wo": n(d, d), "bo": n(d), "ln2_w": 1 + n(d),
        "ln2_b": n(d), "w1": n(f, d), "b1": n(f), "w2": n(d, f), "b2": n(d),
    }


# ----------------------------------------------------------------------------- LayerNorm
def pin_layernorm_hand():
    g = _golden("layernorm_hand.json")
    for c in g["cases"]:
        _close(E.layer_norm(np.array(c["x"], float), c["w"], c["b"], c["eps"]), c["y"], rtol=1e-14, atol=1e-15)


def pin_layernorm_closed_form():
    # With w = 1, b = 0 every row has mean 0 and variance var/(var + eps) exactly.
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 96)) * np.array([[0.01], [0.1], [1], [3], [10], [0.5], [2]]) + 4.0
    eps = 1e-5
    y = E.layer_norm(x, np.ones(96), np.zeros(96), eps)
    var = x.var(axis=-1)
    _close(y.mean(axis=-1), np.zeros(7), atol=1e-12)
    _close((y ** 2).mean(axis=-1), var / (var + eps), rtol=1e-12)


def pin_layernorm_torch():
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(6)
    x, w, b = rng.standard_normal((5, 3, 40)), rng.standard_normal(40), rng.standard_normal(40)
    ref = F.layer_norm(torch.tensor(x), (40,), torch.tensor(w), torch.tensor(b), eps=1e-5).numpy()
    _close(E.layer_norm(x, w, b, 1e-5), ref, rtol=1e-11, atol=1e-12)


# ----------------------------------------------------------------------------- linear
def pin_linear_hand():
    g = _golden("linear_hand.json")
    _close(E.linear(np.array(g["x"], float), np.array(g["w"], float), np.array(g["b"], float)), g["y"])
    # square case: transposing W changes the answer
    w = np.array([[1.0, 2.0], [3.0, 4.0]])
    _close(E.linear(np.array([[1.0, 0.0]]), w, None), [[1.0, 3.0]])


# ----------------------------------------------------------------------------- GELU
def pin_gelu_values():
    g = _golden("gelu_values.json")
    _close(E.gelu(np.array(g["z"], float)), g["y"], rtol=1e-15, atol=1e-16)


def pin_gelu_odd_identity():
    # gelu(z) - gelu(-z) = z * (Phi(z) + Phi(-z)) = z
    z = np.linspace(-6, 6, 241)
    _close(E.gelu(z) - E.gelu(-z), z, rtol=1e-13, atol=1e-14)


def pin_gelu_torch():
    import torch
    import torch.nn.functional as F
    z = np.linspace(-8, 8, 1001)
    _close(E.gelu(z), F.gelu(torch.tensor(z), approximate="none").numpy(), rtol=1e-13, atol=1e-15)


# ----------------------------------------------------------------------------- softmax / attention
def pin_softmax_rows_sum_to_one():
    rng = np.random.default_rng(7)
    s = rng.standard_normal((9, 300)) * 20
    p = E.softmax_rows(s)
    _close(p.sum(axis=-1), np.ones(9), rtol=1e-13)
    assert (p >= 0).all()
    # invariant to a per-row shift, monotone in s
    _close(E.softmax_rows(s + 1000.0), p, rtol=1e-11, atol=1e-300)
    order = np.argsort(s[0])
    assert (np.diff(p[0][order]) >= 0).all()


def pin_attention_hand():
    g = _golden("attention_hand.json")
    c = math.sqrt(2.0) * math.log(3.0)
    q = np.array(g["q_in_units_of_c"], float) * c
    out = E.attention(q, np.array(g["k"], float), np.array(g["v"], float), g["n_heads"])
    _close(out, g["out"], rtol=1e-13, atol=1e-14)


def pin_attention_identical_keys():
    # All keys equal -> every score in a row is equal -> uniform p -> out = mean of V rows.
    rng = np.random.default_rng(8)
    T, H, hd = 257, 3, 8
    q = rng.standard_normal((2, T, H * hd)) * 3
    k = np.broadcast_to(rng.standard_normal((2, 1, H * hd)), (2, T, H * hd))
    v = rng.standard_normal((2, T, H * hd))
    out = E.attention(q, k, v, H)
    _close(out, np.broadcast_to(v.mean(axis=1, keepdims=True), out.shape), rtol=1e-12, atol=1e-13)


def pin_attention_one_hot():
    # One key with a score far above the rest -> out is that key's value row.
    T, H, hd = 50, 2, 4
    rng = np.random.default_rng(9)
    q = np.zeros((T, H * hd)); q[:, 0] = 1.0; q[:, hd] = 1.0
    k = rng.standard_normal((T, H * hd)) * 0.01
    k[17, 0] = 2000.0       # head 0 -> key 17
    k[31, hd] = 2000.0      # head 1 -> key 31
    v = rng.standard_normal((T, H * hd))
    out = E.attention(q, k, v, H)
    _close(out[:, :hd], np.broadcast_to(v[17, :hd], (T, hd)), rtol=1e-12, atol=1e-12)
    _close(out[:, hd:], np.broadcast_to(v[31, hd:], (T, hd)), rtol=1e-12, atol=1e-12)


def pin_attention_online_matches_two_pass():
    rng = np.random.default_rng(10)
    T, H, hd = 300, 2, 16  # three key tiles of 128, the last one ragged (44 keys)
    q, k, v = (rng.standard_normal((2, T, H * hd)) * 2 for _ in range(3))
    _close(E.attention_online(q, k, v, H, tile=128), E.attention(q, k, v, H), rtol=1e-12, atol=1e-12)


def pin_attention_torch_sdpa():
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(11)
    B, T, H, hd = 2, 70, 3, 16
    q, k, v = (rng.standard_normal((B, T, H * hd)) for _ in range(3))
    th = lambda a: torch.tensor(a).reshape(B, T, H, hd).transpose(1, 2)
    ref = F.scaled_dot_product_attention(th(q), th(k), th(v)).transpose(1, 2).reshape(B, T, H * hd).numpy()
    _close(E.attention(q, k, v, H), ref, rtol=1e-11, atol=1e-12)


# ----------------------------------------------------------------------------- block / stack
def _torch_layer(p, n_heads, eps):
    import torch
    import torch.nn as nn
    d = p["wq"].shape[0]
    f = p["w1"].shape[0]
    layer = nn.TransformerEncoderLayer(d, n_heads, f, dropout=0.0, activation="gelu", layer_norm_eps=eps,
                                       batch_first=True, norm_first=True, dtype=torch.float64)
    t = lambda a: torch.tensor(np.asarray(a, np.float64))
    with torch.no_grad():
        layer.self_attn.in_proj_weight.copy_(torch.cat([t(p["wq"]), t(p["wk"]), t(p["wv"])]))
        layer.self_attn.in_proj_bias.copy_(torch.cat([t(p["bq"]), torch.zeros(d, dtype=torch.float64), t(p["bv"])]))
        layer.self_attn.out_proj.weight.copy_(t(p["wo"]))
        layer.self_attn.out_proj.bias.copy_(t(p["bo"]))
        layer.linear1.weight.copy_(t(p["w1"])); layer.linear1.bias.copy_(t(p["b1"]))
        layer.linear2.weight.copy_(t(p["w2"])); layer.linear2.bias.copy_(t(p["b2"]))
        layer.norm1.weight.copy_(t(p["ln1_w"])); layer.norm1.bias.copy_(t(p["ln1_b"]))
        layer.norm2.weight.copy_(t(p["ln2_w"])); layer.norm2.bias.copy_(t(p["ln2_b"]))
    layer.eval()
    return layer


def _torch_run(layers, x):
    import torch
    xt = torch.tensor(np.asarray(x, np.float64)).requires_grad_(True)  # keeps the unfused module path
    y = xt
    for layer in layers:
        y = layer(y)
    return y


def pin_block_hand():
    g = _golden("block_hand.json")
    p = {k: np.array(v, float) for k, v in g["params"].items()}
    x1, y = E.encoder_block(np.array(g["x"], float), p, g["n_heads"], eps=g["eps"], return_mid=True)
    _close(x1, g["x1"], rtol=1e-14, atol=1e-14)
    _close(y, g["y"], rtol=1e-14, atol=1e-14)


def pin_block_zero_weights_is_identity():
    rng = np.random.default_rng(12)
    d, f = 32, 48
    p = {k: np.zeros_like(v) for k, v in _rand_params(rng, d, f).items()}
    p["ln1_w"] = 1 + rng.standard_normal(d); p["ln1_b"] = rng.standard_normal(d)
    p["ln2_w"] = 1 + rng.standard_normal(d); p["ln2_b"] = rng.standard_normal(d)
    x = rng.standard_normal((2, 20, d))
    _close(E.encoder_block(x, p, 4), x, rtol=0, atol=0)


def pin_block_permutation_equivariance():
    rng = np.random.default_rng(13)
    d, f, T = 32, 64, 40
    p = _rand_params(rng, d, f)
    x = rng.standard_normal((T, d))
    perm = rng.permutation(T)
    _close(E.encoder_block(x[perm], p, 4), E.encoder_block(x, p, 4)[perm], rtol=1e-11, atol=1e-12)


def pin_block_torch():
    rng = np.random.default_rng(14)
    d, f, H, T = 32, 80, 4, 37
    p = _rand_params(rng, d, f)
    x = rng.standard_normal((3, T, d))
    ref = _torch_run([_torch_layer(p, H, 1e-5)], x).detach().numpy()
    _close(E.encoder_block(x, p, H, 1e-5), ref, rtol=1e-10, atol=1e-11)


def pin_stack_torch():
    import torch
    rng = np.random.default_rng(15)
    d, f, H, T, L = 24, 40, 3, 29, 3
    layers = [_rand_params(rng, d, f) for _ in range(L)]
    lnf = (1 + rng.standard_normal(d) * 0.3, rng.standard_normal(d) * 0.3)
    x = rng.standard_normal((2, T, d))
    y = _torch_run([_torch_layer(p, H, 1e-5) for p in layers], x)
    ref = torch.nn.functional.layer_norm(y, (d,), torch.tensor(lnf[0]), torch.tensor(lnf[1]), 1e-5).detach().numpy()
    _close(E.encoder_stack(x, layers, H, final=lnf), ref, rtol=1e-10, atol=1e-11)
    ref_nofinal = y.detach().numpy()
    _close(E.encoder_stack(x, layers, H, final=None), ref_nofinal, rtol=1e-10, atol=1e-11)


def pin_block_rows_matches_block():
    rng = np.random.default_rng(16)
    d, f, H, T = 32, 64, 4, 150
    p = _rand_params(rng, d, f)
    x = rng.standard_normal((T, d))
    rows = np.array([0, 5, 77, 149])
    x1, y = E.encoder_block(x, p, H, return_mid=True)
    x1r, yr = E.block_rows(x, rows, p, H)
    _close(x1r, x1[rows], rtol=1e-12, atol=1e-12)
    _close(yr, y[rows], rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- conv stem
def pin_conv1d_hand():
    g = _golden("conv1d_hand.json")
    _close(S.conv1d(g["x"], g["w"], g["b"], stride=1, pad=1), g["y_stride1_pad1"], rtol=1e-14, atol=1e-15)
    _close(S.conv1d(g["x"], g["w"], g["b"], stride=2, pad=1), g["y_stride2_pad1"], rtol=1e-14, atol=1e-15)


def pin_conv1d_closed_forms():
    # One tap per kernel: the centre tap copies the input, the first tap delays it by one
    # frame (zero at t = 0), and stride 2 with the centre tap keeps every other frame.
    rng = np.random.default_rng(11)
    x = rng.standard_normal((2, 9, 4))
    b = rng.standard_normal(4)
    eye = np.eye(4)
    centre = np.zeros((4, 4, 3))
    centre[:, :, 1] = eye
    first = np.zeros((4, 4, 3))
    first[:, :, 0] = eye
    _close(S.conv1d(x, centre, b, 1, 1), x + b)
    delayed = np.concatenate([np.zeros((2, 1, 4)), x[:, :-1]], axis=1)
    _close(S.conv1d(x, first, b, 1, 1), delayed + b)
    _close(S.conv1d(x, centre, b, 2, 1), x[:, ::2] + b)
    # window lengths of the encoder: 3000 mel frames -> 3000 -> 1500 positions
    assert S.conv1d(np.zeros((3000, 1)), np.zeros((1, 1, 3)), [0.0], 1, 1).shape == (3000, 1)
    assert S.conv1d(np.zeros((3000, 1)), np.zeros((1, 1, 3)), [0.0], 2, 1).shape == (1500, 1)


def pin_conv1d_torch():
    import torch
    rng = np.random.default_rng(12)
    x = rng.standard_normal((3, 50, 7))
    w = rng.standard_normal((5, 7, 3))
    b = rng.standard_normal(5)
    for stride in (1, 2):
        ref = torch.nn.functional.conv1d(torch.from_numpy(x).transpose(1, 2), torch.from_numpy(w),
                                         torch.from_numpy(b), stride=stride, padding=1).transpose(1, 2).numpy()
        _close(S.conv1d(x, w, b, stride, 1), ref, rtol=1e-12, atol=1e-12)


def pin_conv_stem_torch():
    # The stem as torch modules: Conv1d(k3, s1, p1) -> exact GELU -> Conv1d(k3, s2, p1) -> exact
    # GELU -> + positions, on one 2-window batch.
    import torch
    rng = np.random.default_rng(13)
    n_mels, d, n = 6, 5, 8
    mel = rng.standard_normal((2, 2 * n, n_mels))
    w1, b1 = rng.standard_normal((d, n_mels, 3)), rng.standard_normal(d)
    w2, b2 = rng.standard_normal((d, d, 3)), rng.standard_normal(d)
    pos = rng.standard_normal((n + 3, d))
    c1 = torch.nn.Conv1d(n_mels, d, 3, stride=1, padding=1).double()
    c2 = torch.nn.Conv1d(d, d, 3, stride=2, padding=1).double()
    with torch.no_grad():
        c1.weight.copy_(torch.from_numpy(w1)); c1.bias.copy_(torch.from_numpy(b1))
        c2.weight.copy_(torch.from_numpy(w2)); c2.bias.copy_(torch.from_numpy(b2))
        gelu = torch.nn.GELU()
        h = gelu(c1(torch.from_numpy(mel).transpose(1, 2)))
        ref = (gelu(c2(h)).transpose(1, 2) + torch.from_numpy(pos[:n])).numpy()
    _close(S.conv_stem(mel, w1, b1, w2, b2, pos), ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- cross K/V
def pin_cross_kv_hand():
    g = _golden("cross_kv_hand.json")
    _close(X.cross_kv(g["enc_out"], g["wk"], g["wv"], g["bv"]), g["kv"], rtol=1e-14, atol=1e-15)


def pin_cross_kv_closed_forms():
    # A zero encoder output gives K = 0 (no K bias) and V = bv in every row; identity weights
    # give K = enc_out and V = enc_out + bv.
    rng = np.random.default_rng(14)
    L, T, d = 3, 5, 4
    wk = rng.standard_normal((L, d, d))
    wv = rng.standard_normal((L, d, d))
    bv = rng.standard_normal((L, d))
    kv = X.cross_kv(np.zeros((T, d)), wk, wv, bv)
    assert kv.shape == (2 * L, T, d)
    _close(kv[0::2], np.zeros((L, T, d)))
    _close(kv[1::2], np.broadcast_to(bv[:, None, :], (L, T, d)))
    x = rng.standard_normal((2, T, d))
    eye = np.broadcast_to(np.eye(d), (L, d, d))
    kv = X.cross_kv(x, eye, eye, bv)
    for l in range(L):
        _close(kv[2 * l], x)
        _close(kv[2 * l + 1], x + bv[l])


def pin_cross_kv_torch():
    import torch
    rng = np.random.default_rng(15)
    L, T, d = 2, 7, 6
    x = rng.standard_normal((T, d))
    wk, wv, bv = rng.standard_normal((L, d, d)), rng.standard_normal((L, d, d)), rng.standard_normal((L, d))
    kv = X.cross_kv(x, wk, wv, bv)
    tx = torch.from_numpy(x)
    for l in range(L):
        _close(kv[2 * l], torch.nn.functional.linear(tx, torch.from_numpy(wk[l])).numpy())
        _close(kv[2 * l + 1], torch.nn.functional.linear(tx, torch.from_numpy(wv[l]), torch.from_numpy(bv[l])).numpy())


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
