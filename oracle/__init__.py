"""Plain float64 CPU oracle of the Whisper encoder's pre-LN transformer blocks.

TEST INFRASTRUCTURE ONLY. Nothing in the product path (the CUDA library and its
Python binding) imports or calls this package; only the tests, the smoke check
and the bench's CPU-baseline leg do. It shares no code with the CUDA path.

Every function is the plain definition of one step, in float64, with numpy /
scipy primitives (matmul, exp, erf) and no blocking, fusion or reordering
beyond what the definition states. Sources, by page and section:

* "inferencelayer 0.2.4 src/whisper_gpu.rs": the ``LN_SRC`` shader (two-pass
  mean and biased variance, eps 1e-5), the ``VANILLA_ATTN`` shader (non-causal
  scaled-dot attention with an online softmax over key tiles of 128) and
  ``WhisperEncoderGpu::forward`` (block order, optional final LN).
* "turbospark-runtime 0.3.0 src/whisper/metal.rs": ``EncLayerGpu`` (no K
  bias), ``encode_layer`` (LN1, Q/K/V, per-head scores scaled by hd^-0.5,
  row softmax, PV, out-proj + add, LN2, fc1, exact-erf GELU, fc2 + add) and
  ``encode_partial`` (stop after n layers, no final norm, for bisection).
* "oxinfer 0.0.5 src/whisper/model.rs": ``WhisperModel::encode`` (the same
  block with ``LN_EPS = 1e-5``, non-causal attention, final ``enc_ln``).

``oracle.stem`` adds the convolutional stem in front of the blocks (conv1 and conv2
with exact-erf GELU, then the positional rows), from turbospark-runtime
``encode_partial`` and oxinfer ``WhisperModel::encode``. ``oracle.cross`` adds the
decoder's cross-attention K/V precompute over the encoder output (inferencelayer's
cross K/V precompute, turbospark-runtime ``build_cross_caches``).

Parity pins live in ``tests/test_oracle_pins.py``: hand-worked cases under
``tests/golden/``, closed forms, invariants and a cross-check against
PyTorch's float64 CPU ``TransformerEncoderLayer`` (norm_first, erf GELU).
"""
from .encoder import (  # noqa: F401
    layer_norm, linear, gelu, softmax_rows, attention, attention_online,
    encoder_block, encoder_stack, block_rows, LN_EPS,
)
from .stem import conv1d, conv_stem  # noqa: F401
from .cross import cross_kv  # noqa: F401
