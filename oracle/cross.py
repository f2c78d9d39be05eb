"""float64 definition of the decoder's cross-attention K/V precompute (test infrastructure only).

Once per window, every decoder layer projects the encoder's output through its cross-attention
key and value weights: K_l = enc_out Wk_l^T (no bias) and V_l = enc_out Wv_l^T + bv_l.
Sources: "inferencelayer 0.2.4 src/whisper_gpu.rs", the cross K/V precompute of its decoder
(one K and one V GEMM per decoder block over the encoder output, no bias); "turbospark-runtime
0.3.0 src/whisper/metal.rs", ``build_cross_caches`` (per decoder layer: K without bias, V with
``cross_v_b``, over ``enc_out``).
"""
from __future__ import annotations

import numpy as np

from .encoder import linear


def cross_kv(enc_out, wk, wv, bv) -> np.ndarray:
    """enc_out [..., T, d]; wk, wv: per-layer [d, d] lists; bv: per-layer [d] list.

    Returns [2 L, ..., T, d]: plane 2l is K of decoder layer l, plane 2l + 1 its V.
    """
    planes = []
    for k_w, v_w, v_b in zip(wk, wv, bv):
        planes.append(linear(enc_out, k_w, None))
        planes.append(linear(enc_out, v_w, v_b))
    return np.stack(planes)
