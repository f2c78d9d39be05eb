"""float64 definition of the encoder's convolutional stem (test infrastructure only).

The stem turns one window of log-mel frames into the encoder's first hidden states:

    h = GELU(conv1(mel))            kernel 3, stride 1, padding 1   (n_mels -> d)
    x = GELU(conv2(h)) + positions  kernel 3, stride 2, padding 1   (d -> d, 2N frames -> N)

Sources: "turbospark-runtime 0.3.0 src/whisper/metal.rs", ``encode_partial`` (the conv front
end: conv1 with stride 1 and padding 1, conv2 with stride 2 and padding 1, exact-erf GELU, then
``transpose_pos`` adds the positional row) and "oxinfer 0.0.5 src/whisper/model.rs",
``WhisperModel::encode`` (conv1 kernel 3 padding 1 then GELU; conv2 kernel 3 stride 2 padding
1, then GELU and the positions). Signals are time-major ``[..., T, C]`` as in oxinfer's
``encode``; weights have the checkpoint layout ``[C_out, C_in, k]``.
"""
from __future__ import annotations

import numpy as np

from .encoder import gelu


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def conv1d(x, w, b, stride: int, pad: int) -> np.ndarray:
    """1-D convolution over time as a neural-network layer computes it (a cross-correlation).

    y[..., t, o] = b[o] + sum_j sum_i w[o, i, j] * x[..., stride*t + j - pad, i]

    with x taken as 0 outside 0 <= index < T_in, for t = 0 .. T_out - 1 where
    T_out = (T_in + 2 pad - k) // stride + 1. x: [..., T_in, C_in]; w: [C_out, C_in, k]; b: [C_out].
    """
    x = _f64(x)
    w = _f64(w)
    c_out, c_in, k = w.shape
    t_in = x.shape[-2]
    if x.shape[-1] != c_in:
        raise ValueError(f"x has {x.shape[-1]} channels, w expects {c_in}")
    t_out = (t_in + 2 * pad - k) // stride + 1
    padding = [(0, 0)] * (x.ndim - 2) + [(pad, pad), (0, 0)]
    xp = np.pad(x, padding)
    y = np.zeros(x.shape[:-2] + (t_out, c_out)) + _f64(b)
    for j in range(k):
        # taps[..., t, i] = x[..., stride*t + j - pad, i]
        taps = xp[..., j: j + stride * (t_out - 1) + 1: stride, :]
        y = y + taps @ w[:, :, j].T
    return y


def conv_stem(mel, conv1_w, conv1_b, conv2_w, conv2_b, positions) -> np.ndarray:
    """mel [..., 2N, n_mels] -> hidden states [..., N, d]: GELU(conv1), GELU(conv2) + positions.

    positions: [>= N, d]; row n is added to output position n.
    """
    h = gelu(conv1d(mel, conv1_w, conv1_b, stride=1, pad=1))
    y = gelu(conv1d(h, conv2_w, conv2_b, stride=2, pad=1))
    return y + _f64(positions)[: y.shape[-2]]
