"""float64 definitions of each step of a Whisper encoder block (test infrastructure only).

Layouts follow the pages: activations are row-major ``[..., T, d]`` with head ``h``
in columns ``h*hd .. (h+1)*hd``; a linear weight is ``[n_out, n_in]`` and computes
``y = x W^T + b``. Every input is widened to float64 before any arithmetic.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf

# oxinfer src/whisper/model.rs, module constants: LN_EPS = 1e-5
# (the LN_SRC shader of inferencelayer src/whisper_gpu.rs adds the same 1e-5).
LN_EPS = 1e-5


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def layer_norm(x, w, b, eps: float = LN_EPS) -> np.ndarray:
    """LayerNorm over the last axis: (x - mean) / sqrt(var + eps) * w + b.

    inferencelayer src/whisper_gpu.rs, ``LN_SRC``: pass one takes the mean, pass two
    the mean of squared deviations (the biased variance, divided by the row width).
    """
    x = _f64(x)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    return (x - mean) / np.sqrt(var + eps) * _f64(w) + _f64(b)


def linear(x, w, b=None) -> np.ndarray:
    """y[n] = sum_k x[k] * W[n, k] + b[n], W stored [n_out, n_in].

    turbospark-runtime src/whisper/metal.rs, ``encode_layer`` (matmul_bias with the
    weight read untransposed); ``b`` is None for the K projection, which has no bias
    (``EncLayerGpu``: "no k bias (openai convention)").
    """
    y = _f64(x) @ _f64(w).T
    if b is not None:
        y = y + _f64(b)
    return y


def gelu(z) -> np.ndarray:
    """Exact (erf) GELU: 0.5 * z * (1 + erf(z / sqrt(2))).

    The pages name it ("exact-erf GELU" in turbospark-runtime ``encode_partial``,
    ``Act::GeluErf`` in inferencelayer ``forward``, ``gelu_erf`` in oxinfer) but do not
    print it; this is the textbook definition z * Phi(z).
    """
    z = _f64(z)
    return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))


def softmax_rows(s) -> np.ndarray:
    """Two-pass softmax over the last axis: p = exp(s - max s) / sum exp(s - max s)."""
    s = _f64(s)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


def _split_heads(a, n_heads: int) -> np.ndarray:
    a = _f64(a)
    *lead, t, d = a.shape
    hd = d // n_heads
    # [..., T, H, hd] -> [..., H, T, hd]
    return np.moveaxis(a.reshape(*lead, t, n_heads, hd), -2, -3)


def _merge_heads(a) -> np.ndarray:
    a = np.moveaxis(a, -3, -2)  # [..., T, H, hd]
    *lead, t, h, hd = a.shape
    return a.reshape(*lead, t, h * hd)


def attention(q, k, v, n_heads: int) -> np.ndarray:
    """Non-causal scaled-dot attention, per window and head, with no mask and no positional term.

    For each head h and query row i: s_j = (q_i . k_j) * hd^-0.5 over every key j of the
    window, p = softmax_j(s), o_i = sum_j p_j v_j, written to the head's column slice.
    Sources: inferencelayer ``VANILLA_ATTN`` (score, softmax, weighted sum) and
    turbospark-runtime ``encode_layer`` (per-head score planes scaled by head_dim^-0.5,
    a row softmax, then scores x V_h into the head's columns).
    q, k, v: [..., T, H*hd]; returns [..., T, H*hd].
    """
    qh, kh, vh = (_split_heads(a, n_heads) for a in (q, k, v))
    hd = qh.shape[-1]
    s = (qh @ np.swapaxes(kh, -1, -2)) * (1.0 / math.sqrt(hd))
    p = softmax_rows(s)
    return _merge_heads(p @ vh)


def attention_online(q, k, v, n_heads: int, tile: int = 128) -> np.ndarray:
    """The same attention computed by the pages' key-tile recurrence (online softmax).

    inferencelayer ``VANILLA_ATTN``: keys are visited in tiles of 128; per tile the
    running maximum m is raised to m' = max(m, max_j s_j), the old denominator and the
    old accumulator are scaled by exp(m - m'), the tile adds sum_j exp(s_j - m') to the
    denominator and sum_j exp(s_j - m') v_j to the accumulator; the output is the
    accumulator divided by the denominator. Used only to pin ``attention``.
    """
    qh, kh, vh = (_split_heads(a, n_heads) for a in (q, k, v))
    hd = qh.shape[-1]
    scale = 1.0 / math.sqrt(hd)
    t_kv = kh.shape[-2]
    run_max = np.full(qh.shape[:-1] + (1,), -np.inf)
    run_den = np.zeros(qh.shape[:-1] + (1,))
    acc = np.zeros(qh.shape)
    for t0 in range(0, t_kv, tile):
        kt = kh[..., t0:t0 + tile, :]
        vt = vh[..., t0:t0 + tile, :]
        s = (qh @ np.swapaxes(kt, -1, -2)) * scale
        new_max = np.maximum(run_max, s.max(axis=-1, keepdims=True))
        corr = np.exp(run_max - new_max)
        p = np.exp(s - new_max)
        run_den = run_den * corr + p.sum(axis=-1, keepdims=True)
        acc = acc * corr + p @ vt
        run_max = new_max
    return _merge_heads(acc / run_den)


def encoder_block(x, p: dict, n_heads: int, eps: float = LN_EPS, return_mid: bool = False):
    """One pre-LN encoder block.

    x1 = x + (attention(LN1(x) Wq^T + bq, LN1(x) Wk^T, LN1(x) Wv^T + bv) Wo^T + bo)
    y  = x1 + (GELU(LN2(x1) W1^T + b1) W2^T + b2)

    Order of steps as in turbospark-runtime ``encode_layer``, inferencelayer
    ``WhisperEncoderGpu::forward`` and oxinfer ``WhisperModel::encode``.
    x: [..., T, d] (one or more windows); attention never mixes windows.
    With ``return_mid`` also returns x1 (the stream after the attention half).
    """
    x = _f64(x)
    h = layer_norm(x, p["ln1_w"], p["ln1_b"], eps)
    q = linear(h, p["wq"], p["bq"])
    k = linear(h, p["wk"], None)
    v = linear(h, p["wv"], p["bv"])
    a = attention(q, k, v, n_heads)
    x1 = x + linear(a, p["wo"], p["bo"])
    h2 = layer_norm(x1, p["ln2_w"], p["ln2_b"], eps)
    u = gelu(linear(h2, p["w1"], p["b1"]))
    y = x1 + linear(u, p["w2"], p["b2"])
    return (x1, y) if return_mid else y


def encoder_stack(x, layers, n_heads: int, final=None, eps: float = LN_EPS) -> np.ndarray:
    """The blocks in order, then the final LayerNorm when ``final = (w, b)`` is given.

    inferencelayer ``forward`` (optional ``ln_post``), turbospark-runtime
    ``encode_partial`` (final layer norm into enc_out), oxinfer ``encode`` (``enc_ln``).
    """
    y = _f64(x)
    for p in layers:
        y = encoder_block(y, p, n_heads, eps)
    if final is not None:
        y = layer_norm(y, final[0], final[1], eps)
    return y


def block_rows(x_window, rows, p: dict, n_heads: int, eps: float = LN_EPS):
    """One block's output for a subset of query rows of ONE window.

    Keys and values need every row of the window, so LN1, K and V run over all of
    ``x_window`` [T, d]; Q, attention, the out projection and the FFN run only for
    ``rows``. Each output row depends on its own input row and on the window's K/V
    alone, so the result equals ``encoder_block(x_window)[rows]``.
    Returns ``(x1_rows, y_rows)``.
    """
    x = _f64(x_window)
    rows = np.asarray(rows)
    h = layer_norm(x, p["ln1_w"], p["ln1_b"], eps)
    k = linear(h, p["wk"], None)
    v = linear(h, p["wv"], p["bv"])
    q = linear(h[rows], p["wq"], p["bq"])
    qh, kh, vh = (_split_heads(a, n_heads) for a in (q, k, v))
    hd = qh.shape[-1]
    s = (qh @ np.swapaxes(kh, -1, -2)) * (1.0 / math.sqrt(hd))
    a = _merge_heads(softmax_rows(s) @ vh)
    x1 = x[rows] + linear(a, p["wo"], p["bo"])
    h2 = layer_norm(x1, p["ln2_w"], p["ln2_b"], eps)
    y = x1 + linear(gelu(linear(h2, p["w1"], p["b1"])), p["w2"], p["b2"])
    return x1, y
