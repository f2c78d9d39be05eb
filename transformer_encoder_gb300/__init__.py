"""wenc: the Whisper encoder's pre-LN transformer blocks on one NVIDIA GB300 (sm_103a).

The compute path is libwenc.so (hand-written CUDA: tcgen05/TMEM GEMMs fed by TMA,
a fused flash-attention kernel, a warp-per-row LayerNorm); ``wenc`` is its ctypes
binding. PyTorch is used only for device memory and streams.
"""
from .wenc import (  # noqa: F401
    WencError, Encoder, attention, attention_tf32, layernorm, linear, linear_tf32, sync_status, selftest_wait_timeout,
    selftest_gemm_pair_abort, selftest_attention_abort,
    gemm_schedule,
    lib, lib_path, EPI_BIAS_BF16, EPI_BIAS_GELU_BF16, EPI_BIAS_RESID_F32, LN_OUT_F32, LN_OUT_BF16, LN_OUT_TF32,
    PREC_BF16, PREC_TF32, EXPORTED_SYMBOLS, LAUNCH_KINDS,
)
