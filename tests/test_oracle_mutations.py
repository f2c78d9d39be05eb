"""Plant plausible mistakes in the oracle (on the CPU) and check that some pin catches each.

A pin set that let one of these through would not prove the oracle right.
"""
import math

import numpy as np
import pytest

import oracle.encoder as E
import oracle.stem as S
import oracle.cross as X
import oracle_pins as P


def _ln_unbiased(x, w, b, eps=E.LN_EPS):
    x = np.asarray(x, np.float64)
    m = x.mean(-1, keepdims=True)
    return (x - m) / np.sqrt(x.var(-1, ddof=1, keepdims=True) + eps) * w + b


def _ln_no_eps(x, w, b, eps=E.LN_EPS):
    x = np.asarray(x, np.float64)
    m = x.mean(-1, keepdims=True)
    return (x - m) / np.sqrt(((x - m) ** 2).mean(-1, keepdims=True)) * w + b


def _ln_no_shift(x, w, b, eps=E.LN_EPS):
    x = np.asarray(x, np.float64)
    m = x.mean(-1, keepdims=True)
    return (x - m) / np.sqrt(((x - m) ** 2).mean(-1, keepdims=True) + eps) * w


def _linear_untransposed(x, w, b=None):
    y = np.asarray(x, np.float64) @ np.asarray(w, np.float64)
    return y if b is None else y + b


def _linear_no_bias(x, w, b=None):
    return np.asarray(x, np.float64) @ np.asarray(w, np.float64).T


def _gelu_tanh(z):
    z = np.asarray(z, np.float64)
    return 0.5 * z * (1 + np.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3)))


def _attention_scale_hd(q, k, v, n_heads):
    qh, kh, vh = (E._split_heads(a, n_heads) for a in (q, k, v))
    s = (qh @ np.swapaxes(kh, -1, -2)) / qh.shape[-1]
    return E._merge_heads(E.softmax_rows(s) @ vh)


def _attention_wrong_axis(q, k, v, n_heads):
    qh, kh, vh = (E._split_heads(a, n_heads) for a in (q, k, v))
    s = (qh @ np.swapaxes(kh, -1, -2)) / math.sqrt(qh.shape[-1])
    p = np.swapaxes(E.softmax_rows(np.swapaxes(s, -1, -2)), -1, -2)
    return E._merge_heads(p @ vh)


def _attention_heads_interleaved(q, k, v, n_heads):
    def split(a):
        a = np.asarray(a, np.float64)
        *lead, t, d = a.shape
        return np.moveaxis(a.reshape(*lead, t, d // n_heads, n_heads), -1, -3)
    qh, kh, vh = split(q), split(k), split(v)
    s = (qh @ np.swapaxes(kh, -1, -2)) / math.sqrt(qh.shape[-1])
    o = E.softmax_rows(s) @ vh  # [..., H, T, hd]
    o = np.moveaxis(o, -3, -1)  # [..., T, hd, H]
    *lead, t, hd, h = o.shape
    return o.reshape(*lead, t, hd * h)


def _softmax_no_max(s):
    e = np.exp(np.asarray(s, np.float64) - 1.0)
    return e / (e.sum(-1, keepdims=True) + 1e-3)


def _block_variant(kind):
    def block(x, p, n_heads, eps=E.LN_EPS, return_mid=False):
        x = np.asarray(x, np.float64)
        h = E.layer_norm(x, p["ln1_w"], p["ln1_b"], eps)
        q = E.linear(h, p["wq"], p["bq"])
        k = E.linear(h, p["wq"] if kind == "k_uses_wq" else p["wk"], None)
        v = E.linear(h, p["wv"], None if kind == "v_drops_bias" else p["bv"])
        a = E.attention(q, k, v, n_heads)
        x1 = x + E.linear(a, p["wo"], p["bo"])
        src = x if kind == "ln2_on_x" else x1
        ln2 = ("ln1_w", "ln1_b") if kind == "ln1_params_twice" else ("ln2_w", "ln2_b")
        h2 = E.layer_norm(src, p[ln2[0]], p[ln2[1]], eps)
        u = E.linear(h2, p["w1"], p["b1"])
        u = u if kind == "no_gelu" else E.gelu(u)
        f = E.linear(u, p["w2"], p["b2"])
        y = f if kind == "no_ffn_residual" else x1 + f
        return (x1, y) if return_mid else y
    return block


def _stack_drops_final(x, layers, n_heads, final=None, eps=E.LN_EPS):
    y = np.asarray(x, np.float64)
    for p in layers:
        y = E.encoder_block(y, p, n_heads, eps)
    return y


def _conv_flipped(x, w, b, stride, pad):
    # a true convolution (kernel reversed) instead of the layer's cross-correlation
    return _CONV(x, np.asarray(w, np.float64)[:, :, ::-1], b, stride, pad)


def _conv_channels_swapped(x, w, b, stride, pad):
    w = np.asarray(w, np.float64)
    return _CONV(x, np.swapaxes(w, 0, 1) if w.shape[0] == w.shape[1] else w, b, stride, pad)


def _conv_pad_right_only(x, w, b, stride, pad):
    # all the padding after the window: taps at t, t+1, t+2 instead of t-1, t, t+1
    x = np.asarray(x, np.float64)
    xp = np.concatenate([x, np.zeros(x.shape[:-2] + (2 * pad, x.shape[-1]))], axis=-2)
    return _CONV(xp, w, b, stride, 0)


def _stem_variant(kind):
    def stem(mel, w1, b1, w2, b2, positions):
        h = E.gelu(S.conv1d(mel, w1, b1, stride=2 if kind == "conv1_strided" else 1, pad=1))
        y = S.conv1d(h, w2, b2, stride=2, pad=1)
        pos = np.asarray(positions, np.float64)[: y.shape[-2]]
        if kind == "gelu_after_positions":
            return E.gelu(y + pos)
        y = E.gelu(y)
        return y if kind == "no_positions" else y + pos
    return stem


_CONV = S.conv1d


def _cross_variant(kind):
    def cross(enc_out, wk, wv, bv):
        planes = []
        for k_w, v_w, v_b in zip(wk, wv, bv):
            k = E.linear(enc_out, k_w, v_b if kind == "k_gets_v_bias" else None)
            v = E.linear(enc_out, v_w, v_b)
            planes += [v, k] if kind == "kv_swapped" else [k, v]
        return np.stack(planes)
    return cross

MUTATIONS = {
    "ln_unbiased_variance": ("layer_norm", _ln_unbiased),
    "ln_missing_eps": ("layer_norm", _ln_no_eps),
    "ln_missing_shift": ("layer_norm", _ln_no_shift),
    "linear_untransposed": ("linear", _linear_untransposed),
    "linear_drops_bias": ("linear", _linear_no_bias),
    "gelu_tanh_approx": ("gelu", _gelu_tanh),
    "attn_scale_1_over_hd": ("attention", _attention_scale_hd),
    "attn_softmax_over_queries": ("attention", _attention_wrong_axis),
    "attn_heads_interleaved": ("attention", _attention_heads_interleaved),
    "softmax_unnormalised": ("softmax_rows", _softmax_no_max),
    # (A K bias is not listed: it adds q.b to every score of a row, which the softmax
    # cancels, so it is not a mistake the output can show.)
    "block_k_uses_wq": ("encoder_block", _block_variant("k_uses_wq")),
    "block_v_drops_bias": ("encoder_block", _block_variant("v_drops_bias")),
    "block_ln2_on_x": ("encoder_block", _block_variant("ln2_on_x")),
    "block_ln1_params_twice": ("encoder_block", _block_variant("ln1_params_twice")),
    "block_no_gelu": ("encoder_block", _block_variant("no_gelu")),
    "block_no_ffn_residual": ("encoder_block", _block_variant("no_ffn_residual")),
    "stack_drops_final_ln": ("encoder_stack", _stack_drops_final),
    "conv_kernel_flipped": ("S.conv1d", _conv_flipped),
    "conv_channels_swapped": ("S.conv1d", _conv_channels_swapped),
    "conv_padding_one_sided": ("S.conv1d", _conv_pad_right_only),
    "stem_no_positions": ("S.conv_stem", _stem_variant("no_positions")),
    "stem_gelu_after_positions": ("S.conv_stem", _stem_variant("gelu_after_positions")),
    "stem_conv1_strided": ("S.conv_stem", _stem_variant("conv1_strided")),
    "cross_k_gets_v_bias": ("X.cross_kv", _cross_variant("k_gets_v_bias")),
    "cross_kv_planes_swapped": ("X.cross_kv", _cross_variant("kv_swapped")),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    module = E
    if attr.startswith("S."):
        module, attr = S, attr[2:]
    elif attr.startswith("X."):
        module, attr = X, attr[2:]
    monkeypatch.setattr(module, attr, fn)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
