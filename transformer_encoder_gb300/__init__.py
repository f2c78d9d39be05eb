"""wenc: the Whisper encoder's pre-LN transformer blocks on one NVIDIA GB300 (sm_103a).

The compute path is libwenc.so (hand-written CUDA: tcgen05/TMEM GEMMs fed by TMA,
a fused flash-attention kernel, a warp-per-row LayerNorm); ``wenc`` is its ctypes
binding. PyTorch is used only for device memory and streams.
"""
from .wenc import (  # noqa: F401
    WencError, Encoder, attention, layernorm, linear, sync_status, selftest_wait_timeout, lib, lib_path,
    EPI_BIAS_BF16, EPI_BIAS_GELU_BF16, EPI_BIAS_RESID_F32, EXPORTED_SYMBOLS, LAUNCH_KINDS,
)
