"""Seeded synthetic inputs for the Whisper encoder blocks.

This module only draws random numbers and stores them; it holds none of the
encoder's arithmetic. Both the f64 oracle (through the tests and the bench's
CPU leg) and the CUDA path read what it produces, so the two sides always see
the same weights and hidden states.

Recipe (one ``numpy.random.Generator(PCG64(seed))`` per workload, drawn in
float32, in this fixed order):

  for each layer:  ln1_w, ln1_b, wq, bq, wk, wv, bv, wo, bo,
                   ln2_w, ln2_b, w1, b1, w2, b2
  then:            lnf_w, lnf_b          (drawn even when the final LN is off)
  then:            x  ~ N(0, 1)   [B, T, d]

  weight matrices  ~ N(0, 0.02), stored [n_out, n_in] (PyTorch layout)
  biases           ~ N(0, 0.01)   (the K projection has none)
  LN scale         = 1 + N(0, 0.02),  LN shift ~ N(0, 0.02)

Workloads whose weights are declared bf16 have every weight matrix rounded
to bfloat16 (round to nearest, ties to even) right after it is drawn; norms
and biases stay float32. The dimensions are Whisper tiny / base / small /
large-v3; no checkpoint or audio is read.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "LAYER_KEYS", "MATRIX_KEYS",
    "f32_to_bf16_bits", "bf16_bits_to_f32", "round_to_bf16", "round_to_tf32",
    "make_layer", "make_weights", "make_input", "make_qkv", "make_stem", "make_mel", "make_cross",
]

T_WINDOW = 1500  # encoder positions of one zero-padded 30 s window

LAYER_KEYS = ("ln1_w", "ln1_b", "wq", "bq", "wk", "wv", "bv", "wo", "bo",
              "ln2_w", "ln2_b", "w1", "b1", "w2", "b2")
MATRIX_KEYS = ("wq", "wk", "wv", "wo", "w1", "w2")


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    d_model: int
    n_heads: int
    ffn_dim: int
    n_layers: int
    final_ln: bool
    bf16_weights: bool
    seq_len: int = T_WINDOW
    seed: int = 0
    head_dim: int = field(default=64)
    n_mels: int = 80  # mel bands of the convolutional stem's input (128 for large-v3)

    @property
    def rows(self) -> int:
        return self.batch * self.seq_len

    def flops(self) -> float:
        """Dense FLOPs of one call: four projections, two FFN GEMMs, QK^T and PV."""
        d, f, T, B = self.d_model, self.ffn_dim, self.seq_len, self.batch
        per_layer = 2.0 * B * T * (4 * d * d + 2 * d * f) + 4.0 * B * self.n_heads * T * T * self.head_dim
        return self.n_layers * per_layer


WORKLOADS = {
    "tiny_block": Workload("tiny_block", 1, 384, 6, 1536, 1, final_ln=False, bf16_weights=False),
    "tiny_stack": Workload("tiny_stack", 1, 384, 6, 1536, 4, final_ln=True, bf16_weights=True),
    "base_stack": Workload("base_stack", 4, 512, 8, 2048, 6, final_ln=True, bf16_weights=True),
    "small_stack": Workload("small_stack", 8, 768, 12, 3072, 12, final_ln=True, bf16_weights=True),
    "large_stack": Workload("large_stack", 16, 1280, 20, 5120, 32, final_ln=True, bf16_weights=True, n_mels=128),
    # One block at large-v3 dims and batch 16: every kernel launch has exactly the shape it has
    # inside the 32-block stack, with ~1 GB on the device (used for profiler captures).
    "large_block": Workload("large_block", 16, 1280, 20, 5120, 1, final_ln=True, bf16_weights=True, n_mels=128),
    # Two such blocks: the first block's fc2 also writes the row statistics and bf16 copy the
    # second block's QKV reads, as every block but the last does in the 32-block stack.
    "large_pair": Workload("large_pair", 16, 1280, 20, 5120, 2, final_ln=True, bf16_weights=True, n_mels=128),
}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the raw 16-bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """float32 array whose values are exactly representable in bfloat16."""
    return bf16_bits_to_f32(f32_to_bf16_bits(a))


def round_to_tf32(a: np.ndarray) -> np.ndarray:
    """float32 array rounded to TF32 (10 explicit mantissa bits), nearest with ties away from
    zero: the values a TF32 tensor-core operand holds exactly (finite inputs only)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x1000) & 0xFFFFE000
    return u.astype(np.uint32).view(np.float32)


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def make_layer(rng: np.random.Generator, d: int, f: int, bf16: bool) -> dict:
    """Draw one block's parameters in the fixed order. Matrices are [n_out, n_in] float32."""
    mat = (lambda shape: round_to_bf16(_normal(rng, shape, 0.02))) if bf16 else (lambda shape: _normal(rng, shape, 0.02))
    p = {}
    p["ln1_w"] = (1.0 + _normal(rng, (d,), 0.02)).astype(np.float32)
    p["ln1_b"] = _normal(rng, (d,), 0.02)
    p["wq"] = mat((d, d))
    p["bq"] = _normal(rng, (d,), 0.01)
    p["wk"] = mat((d, d))
    p["wv"] = mat((d, d))
    p["bv"] = _normal(rng, (d,), 0.01)
    p["wo"] = mat((d, d))
    p["bo"] = _normal(rng, (d,), 0.01)
    p["ln2_w"] = (1.0 + _normal(rng, (d,), 0.02)).astype(np.float32)
    p["ln2_b"] = _normal(rng, (d,), 0.02)
    p["w1"] = mat((f, d))
    p["b1"] = _normal(rng, (f,), 0.01)
    p["w2"] = mat((d, f))
    p["b2"] = _normal(rng, (d,), 0.01)
    return p


def make_weights(w: Workload, rng: np.random.Generator | None = None, layer_callback=None):
    """All parameters of a workload, drawn from a fresh generator seeded with ``w.seed``.

    Returns ``(layers, final, rng)``: ``layers`` is a list of per-block dicts (or, when
    ``layer_callback`` is given, the list of whatever it returns for each freshly drawn
    block, so that large stacks need not stay in host memory), ``final`` is ``(lnf_w, lnf_b)``
    and ``rng`` is the generator positioned to draw the input next.
    """
    if rng is None:
        rng = np.random.Generator(np.random.PCG64(w.seed))
    layers = []
    for _ in range(w.n_layers):
        p = make_layer(rng, w.d_model, w.ffn_dim, w.bf16_weights)
        layers.append(layer_callback(p) if layer_callback is not None else p)
    lnf_w = (1.0 + _normal(rng, (w.d_model,), 0.02)).astype(np.float32)
    lnf_b = _normal(rng, (w.d_model,), 0.02)
    return layers, (lnf_w, lnf_b), rng


def make_input(w: Workload, rng: np.random.Generator, batch: int | None = None) -> np.ndarray:
    """Hidden states [B, T, d] ~ N(0, 1), float32 (drawn after all parameters)."""
    b = w.batch if batch is None else batch
    return rng.standard_normal((b, w.seq_len, w.d_model), dtype=np.float32)


STEM_SEED_OFFSET = 7919  # the stem draws from a generator of its own (block draws unchanged)


def make_stem(w: Workload) -> dict:
    """Convolutional-stem parameters: conv1_w [d, n_mels, 3], conv2_w [d, d, 3] (checkpoint
    layout), conv biases [d], and the positional table [seq_len, d].

    Matrices ~ N(0, 0.02) (rounded to bf16 for bf16 workloads), biases ~ N(0, 0.01), positions
    ~ U(-1, 1) (the value range of Whisper's sinusoidal table), from PCG64(seed + 7919).
    """
    rng = np.random.Generator(np.random.PCG64(w.seed + STEM_SEED_OFFSET))
    mat = (lambda shape: round_to_bf16(_normal(rng, shape, 0.02))) if w.bf16_weights else (lambda shape: _normal(rng, shape, 0.02))
    d = w.d_model
    p = {}
    p["conv1_w"] = mat((d, w.n_mels, 3))
    p["conv1_b"] = _normal(rng, (d,), 0.01)
    p["conv2_w"] = mat((d, d, 3))
    p["conv2_b"] = _normal(rng, (d,), 0.01)
    p["positions"] = rng.uniform(-1.0, 1.0, (w.seq_len, d)).astype(np.float32)
    return p


CROSS_SEED_OFFSET = 104729  # the decoder's cross K/V weights draw from a generator of their own


def make_cross(w: Workload, n_dec: int | None = None) -> list:
    """Decoder cross-attention K/V weights, one dict per decoder layer (n_dec defaults to the
    encoder's layer count, as in every Whisper size): wk, wv [d, d] ~ N(0, 0.02) (rounded to
    bf16 for bf16 workloads), bv [d] ~ N(0, 0.01), from PCG64(seed + 104729)."""
    rng = np.random.Generator(np.random.PCG64(w.seed + CROSS_SEED_OFFSET))
    mat = (lambda shape: round_to_bf16(_normal(rng, shape, 0.02))) if w.bf16_weights else (lambda shape: _normal(rng, shape, 0.02))
    d = w.d_model
    out = []
    for _ in range(w.n_layers if n_dec is None else n_dec):
        out.append({"wk": mat((d, d)), "wv": mat((d, d)), "bv": _normal(rng, (d,), 0.01)})
    return out


def make_mel(w: Workload, batch: int | None = None, seed: int = 2) -> np.ndarray:
    """Log-mel windows [B, 2 * seq_len, n_mels] (time-major), ~ U(-1, 1): the range of Whisper's
    normalised log-mel features."""
    rng = np.random.Generator(np.random.PCG64(seed))
    b = w.batch if batch is None else batch
    return rng.uniform(-1.0, 1.0, (b, 2 * w.seq_len, w.n_mels)).astype(np.float32)


def make_qkv(batch: int, seq: int, heads: int, head_dim: int = 64, seed: int = 1, scale: float = 1.0):
    """q, k, v as bf16 bit patterns [B, T, H, hd], values ~ N(0, scale^2) rounded to bf16.

    ``scale`` = 1 gives the sharp softmax of the standalone attention sweep; 0.1 a soft one.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for _ in range(3):
        a = _normal(rng, (batch, seq, heads, head_dim), scale)
        out.append(f32_to_bf16_bits(a))
    return tuple(out)
