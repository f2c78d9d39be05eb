"""Thin ctypes binding of libwenc.so (argument marshalling only).

Every step of the encoder runs in the library's CUDA kernels; this module only turns
PyTorch tensors (used here for device memory and streams) into the pointers and sizes
of the C ABI declared in include/wenc.h, and turns non-OK statuses into exceptions.
There is no fallback: if the library is missing or the device is not sm_103a, calls raise.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "WencError", "lib", "lib_path", "Encoder", "attention", "attention_tf32", "layernorm", "linear", "linear_tf32",
    "sync_status", "selftest_gemm_pair_abort", "EPI_BIAS_BF16", "EPI_BIAS_GELU_BF16", "EPI_BIAS_RESID_F32", "LN_OUT_F32", "LN_OUT_BF16",
    "LN_OUT_TF32", "PREC_BF16", "PREC_TF32", "EXPORTED_SYMBOLS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
# WENC_LIBRARY may name another library built in-tree into _lib/ (the index-checked
# libwenc_bounds.so); anything outside _lib/ is refused.
lib_path = os.path.join(_PKG, "_lib", os.path.basename(os.environ.get("WENC_LIBRARY") or "libwenc.so"))

EPI_BIAS_BF16, EPI_BIAS_GELU_BF16, EPI_BIAS_RESID_F32 = 0, 1, 2
LN_OUT_F32, LN_OUT_BF16, LN_OUT_TF32 = 0, 1, 2
PREC_BF16, PREC_TF32 = 0, 1
_STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "OOM", 4: "CUDA", 5: "DEVICE_TIMEOUT"}
LAUNCH_KINDS = {0: "layernorm", 1: "gemm_qkv", 2: "attention", 3: "gemm_out", 4: "gemm_fc1", 5: "gemm_fc2",
                6: "layernorm_final", 7: "copy", 8: "attention_combine", 9: "stem_unfold", 10: "gemm_conv1",
                11: "gemm_conv2", 12: "cross_kv_cast", 13: "gemm_cross_kv", 14: "row_stats"}

EXPORTED_SYMBOLS = (
    "wenc_create", "wenc_forward", "wenc_forward_layers", "wenc_forward_launches", "wenc_set_launch_events",
    "wenc_attention", "wenc_layernorm", "wenc_linear", "wenc_sync_status", "wenc_destroy", "wenc_last_error",
    "wenc_version", "wenc_selftest_wait_timeout", "wenc_attention_static", "wenc_attention_static_capacity",
    "wenc_linear_tf32", "wenc_attention_tf32", "wenc_set_stem", "wenc_stem", "wenc_encode", "wenc_encode_launches",
    "wenc_set_cross_kv", "wenc_cross_kv", "wenc_selftest_gemm_schedule", "wenc_selftest_gemm_pair_abort",
    "wenc_set_device_alloc_limit", "wenc_device_bytes_held", "wenc_selftest_attention_abort",
)


class WencError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"wenc {_STATUS.get(status, status)}: {message}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("d_model", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("ffn_dim", ctypes.c_int), ("seq_len", ctypes.c_int),
                ("max_batch", ctypes.c_int), ("final_ln", ctypes.c_int), ("ln_eps", ctypes.c_float),
                ("weight_dtype", ctypes.c_int), ("precision", ctypes.c_int)]


_LW_FIELDS = ("ln1_w", "ln1_b", "wq", "bq", "wk", "bk", "wv", "bv", "wo", "bo", "ln2_w", "ln2_b", "w1", "b1", "w2", "b2")


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _LW_FIELDS]


STEM_KEYS = ("conv1_w", "conv1_b", "conv2_w", "conv2_b", "positions")


class StemWeights(ctypes.Structure):
    _fields_ = [("n_mels", ctypes.c_int)] + [(n, ctypes.c_void_p) for n in STEM_KEYS]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libwenc.so (built in-tree by transformer_encoder_gb300.build); raise if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(lib_path):
            raise RuntimeError(f"{lib_path} is missing: build it with `python -m transformer_encoder_gb300.build`")
        L = ctypes.CDLL(lib_path)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.wenc_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(LayerWeights), vp, vp, vp, ctypes.POINTER(vp)]
        L.wenc_forward.argtypes = [vp, vp, vp, i, vp]
        L.wenc_forward_layers.argtypes = [vp, vp, vp, i, i, i, i, vp]
        L.wenc_forward_launches.argtypes = [vp, i, i, i]
        L.wenc_set_launch_events.argtypes = [vp, ctypes.POINTER(vp), i, ctypes.POINTER(i)]
        L.wenc_attention.argtypes = [vp, vp, vp, vp, i, i, i, i, vp]
        L.wenc_layernorm.argtypes = [vp, vp, vp, vp, i, i, f, i, vp]
        L.wenc_linear.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, vp]
        L.wenc_linear_tf32.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, vp]
        L.wenc_set_stem.argtypes = [vp, ctypes.POINTER(StemWeights), vp]
        L.wenc_stem.argtypes = [vp, vp, vp, i, vp]
        L.wenc_encode.argtypes = [vp, vp, vp, i, vp]
        L.wenc_encode_launches.argtypes = [vp]
        L.wenc_set_cross_kv.argtypes = [vp, i, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp), vp]
        L.wenc_cross_kv.argtypes = [vp, vp, vp, i, vp]
        L.wenc_attention_tf32.argtypes = [vp, vp, vp, vp, i, i, i, i, vp]
        L.wenc_sync_status.argtypes = [vp]
        L.wenc_selftest_wait_timeout.argtypes = [vp]
        L.wenc_selftest_gemm_pair_abort.argtypes = [vp, vp, vp, vp, i, i, i, i, vp]
        L.wenc_selftest_attention_abort.argtypes = [vp, vp, vp, vp, i, i, i, i, vp]
        L.wenc_set_device_alloc_limit.argtypes = [ctypes.c_size_t]
        L.wenc_set_device_alloc_limit.restype = None
        L.wenc_device_bytes_held.argtypes = []
        L.wenc_device_bytes_held.restype = ctypes.c_size_t
        ip = ctypes.POINTER(ctypes.c_int)
        L.wenc_selftest_gemm_schedule.argtypes = [i, i, i, i, ip, i, ip, ip, ip]
        L.wenc_attention_static.argtypes = [vp, vp, vp, vp, i, i, i, i, vp]
        L.wenc_attention_static.restype = ctypes.c_int
        L.wenc_attention_static_capacity.argtypes = []
        L.wenc_attention_static_capacity.restype = ctypes.c_size_t
        L.wenc_destroy.argtypes = [vp]
        L.wenc_destroy.restype = None
        L.wenc_last_error.restype = ctypes.c_char_p
        L.wenc_version.restype = ctypes.c_char_p
        for name in ("wenc_create", "wenc_forward", "wenc_forward_layers", "wenc_set_launch_events", "wenc_attention",
                     "wenc_layernorm", "wenc_linear", "wenc_sync_status", "wenc_forward_launches",
                     "wenc_selftest_wait_timeout", "wenc_linear_tf32", "wenc_attention_tf32", "wenc_set_stem",
                     "wenc_stem", "wenc_encode", "wenc_encode_launches", "wenc_set_cross_kv", "wenc_cross_kv",
                     "wenc_selftest_gemm_schedule", "wenc_selftest_gemm_pair_abort", "wenc_selftest_attention_abort"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int):
    if status != 0:
        raise WencError(status, lib().wenc_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _require(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class Encoder:
    """A wenc handle: packed resident weights plus a workspace for `max_batch` windows.

    ``layers`` is a list of dicts with the keys of ``synth.LAYER_KEYS`` holding CUDA tensors
    (matrices float32 or bfloat16 [n_out, n_in], vectors float32). The library copies and
    packs them, so they may be freed after construction. ``precision`` is "bf16" (bf16
    tensor-core operands) or "tf32" (TF32 operands, fp32 activations).
    """

    def __init__(self, layers, n_heads: int, seq_len: int, max_batch: int, final=None, ln_eps: float = 1e-5,
                 stream=None, precision: str = "bf16"):
        import torch
        L = lib()
        d = layers[0]["wq"].shape[0]
        f = layers[0]["w1"].shape[0]
        mdtype = layers[0]["wq"].dtype
        if mdtype not in (torch.float32, torch.bfloat16):
            raise TypeError("weight matrices must be float32 or bfloat16")
        if precision not in ("bf16", "tf32"):
            raise ValueError(f"precision must be 'bf16' or 'tf32', got {precision!r}")
        cfg = Config(len(layers), d, n_heads, d // n_heads, f, seq_len, max_batch, 1 if final is not None else 0,
                     ln_eps, 1 if mdtype == torch.bfloat16 else 0, PREC_TF32 if precision == "tf32" else PREC_BF16)
        self.precision = precision
        self.n_dec = 0  # decoder layers of the cross K/V weights (set_cross_kv)
        arr = (LayerWeights * len(layers))()
        for i, p in enumerate(layers):
            for k in ("wq", "wk", "wv", "wo", "w1", "w2"):
                _require(p[k], mdtype, k)
            for k in ("ln1_w", "ln1_b", "bq", "bv", "bo", "ln2_w", "ln2_b", "b1", "b2"):
                _require(p[k], torch.float32, k)
            for k in _LW_FIELDS:
                setattr(arr[i], k, None if k == "bk" else p[k].data_ptr())
        lnf_w = lnf_b = None
        if final is not None:
            _require(final[0], torch.float32, "lnf_w")
            _require(final[1], torch.float32, "lnf_b")
            lnf_w, lnf_b = _ptr(final[0]), _ptr(final[1])
        h = ctypes.c_void_p()
        _check(L.wenc_create(ctypes.byref(cfg), arr, lnf_w, lnf_b, _stream(stream), ctypes.byref(h)))
        self._h = h
        self.cfg = cfg
        self.d_model, self.ffn_dim, self.n_layers, self.seq_len, self.max_batch = d, f, len(layers), seq_len, max_batch

    @property
    def handle(self):
        return self._h

    def forward(self, x, out=None, stream=None):
        """out = Encoder(x), x float32 CUDA [B, seq_len, d]; out may be x (in place)."""
        return self.forward_layers(x, out, 0, self.n_layers, True, stream)

    def forward_layers(self, x, out=None, first: int = 0, count: int | None = None, final_ln: bool = True,
                       stream=None):
        import torch
        _require(x, torch.float32, "x")
        if count is None:
            count = self.n_layers - first
        if out is None:
            out = torch.empty_like(x)
        _require(out, torch.float32, "out")
        B = x.shape[0]
        _check(lib().wenc_forward_layers(self._h, _ptr(x), _ptr(out), B, first, count, int(final_ln), _stream(stream)))
        return out

    def set_stem(self, stem: dict, stream=None):
        """Attach the convolutional stem: ``stem`` has the keys of ``STEM_KEYS`` as CUDA tensors
        (conv weights [d, C_in, 3] in the layers' matrix dtype, biases [d] and positions
        [seq_len, d] float32); n_mels is read from conv1_w."""
        import torch
        mdtype = torch.bfloat16 if self.cfg.weight_dtype == 1 else torch.float32
        _require(stem["conv1_w"], mdtype, "conv1_w")
        _require(stem["conv2_w"], mdtype, "conv2_w")
        for k in ("conv1_b", "conv2_b", "positions"):
            _require(stem[k], torch.float32, k)
        self.n_mels = int(stem["conv1_w"].shape[1])
        w = StemWeights(self.n_mels, *[stem[k].data_ptr() for k in STEM_KEYS])
        _check(lib().wenc_set_stem(self._h, ctypes.byref(w), _stream(stream)))

    def stem(self, mel, out=None, stream=None):
        """hidden [B, seq_len, d] = stem(mel), mel float32 CUDA [B, 2*seq_len, n_mels]."""
        import torch
        _require(mel, torch.float32, "mel")
        if out is None:
            out = torch.empty((mel.shape[0], self.seq_len, self.d_model), dtype=torch.float32, device=mel.device)
        _require(out, torch.float32, "out")
        _check(lib().wenc_stem(self._h, _ptr(mel), _ptr(out), mel.shape[0], _stream(stream)))
        return out

    def encode(self, mel, out=None, stream=None):
        """The whole encoder from log-mel frames: stem, blocks and the final LayerNorm."""
        import torch
        _require(mel, torch.float32, "mel")
        if out is None:
            out = torch.empty((mel.shape[0], self.seq_len, self.d_model), dtype=torch.float32, device=mel.device)
        _require(out, torch.float32, "out")
        _check(lib().wenc_encode(self._h, _ptr(mel), _ptr(out), mel.shape[0], _stream(stream)))
        return out

    def set_cross_kv(self, dec_layers, stream=None):
        """Attach the decoder's cross-attention K/V weights: a list (one per decoder layer) of
        dicts with wk, wv ([d, d], the layers' matrix dtype) and bv ([d] float32) CUDA tensors."""
        import torch
        mdtype = torch.bfloat16 if self.cfg.weight_dtype == 1 else torch.float32
        n = len(dec_layers)
        for p in dec_layers:
            _require(p["wk"], mdtype, "wk")
            _require(p["wv"], mdtype, "wv")
            _require(p["bv"], torch.float32, "bv")
        arr = lambda key: (ctypes.c_void_p * n)(*[p[key].data_ptr() for p in dec_layers])
        wk, wv, bv = arr("wk"), arr("wv"), arr("bv")
        _check(lib().wenc_set_cross_kv(self._h, n, wk, wv, bv, _stream(stream)))
        self.n_dec = n

    def cross_kv(self, enc_out, out=None, stream=None):
        """[2 n_dec, B * seq_len, d] cross K/V planes (K of layer l at 2l, V at 2l + 1) of an
        encoder output float32 [B, seq_len, d]; bf16 for the bf16 precision, float32 for TF32."""
        import torch
        _require(enc_out, torch.float32, "enc_out")
        B = enc_out.shape[0]
        dt = torch.float32 if self.precision == "tf32" else torch.bfloat16
        if self.n_dec == 0:  # the library reports the missing weights
            _check(lib().wenc_cross_kv(self._h, _ptr(enc_out), None, B, _stream(stream)))
        if out is None:
            out = torch.empty((2 * self.n_dec, B * self.seq_len, self.d_model), dtype=dt, device=enc_out.device)
        _require(out, dt, "out")
        _check(lib().wenc_cross_kv(self._h, _ptr(enc_out), _ptr(out), B, _stream(stream)))
        return out

    def encode_launches(self) -> int:
        return lib().wenc_encode_launches(self._h)

    def launches(self, first: int = 0, count: int | None = None, final_ln: bool = True) -> int:
        count = self.n_layers - first if count is None else count
        return lib().wenc_forward_launches(self._h, first, count, int(final_ln))

    def set_launch_events(self, events, want_kinds: bool = True):
        """Arm the per-launch timing hook for the next forward call (torch.cuda.Event list)."""
        n = len(events)
        ev = (ctypes.c_void_p * n)(*[e.cuda_event for e in events])
        kinds = (ctypes.c_int * n)() if want_kinds else None
        self._ev_keep = (ev, kinds)
        _check(lib().wenc_set_launch_events(self._h, ev, n, kinds))
        return kinds

    def sync_status(self):
        _check(lib().wenc_sync_status(self._h))

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().wenc_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def attention(q, k, v, out=None, stream=None):
    """out = softmax(q k^T / 8) v per (window, head); q, k, v bf16 CUDA [B, T, H, 64]."""
    import torch
    for n, t in (("q", q), ("k", k), ("v", v)):
        _require(t, torch.bfloat16, n)
    B, T, H, hd = q.shape
    if out is None:
        out = torch.empty_like(q)
    _require(out, torch.bfloat16, "out")
    _check(lib().wenc_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, T, H, hd, _stream(stream)))
    return out


def layernorm(x, w, b, eps: float = 1e-5, out_bf16: bool = True, out=None, stream=None, out_format=None):
    """LayerNorm over the last axis of a float32 CUDA tensor.

    Output bf16 (``out_bf16``) or float32; ``out_format`` (LN_OUT_*) overrides it and also
    offers float32 rounded to TF32.
    """
    import torch
    _require(x, torch.float32, "x")
    fmt = (LN_OUT_BF16 if out_bf16 else LN_OUT_F32) if out_format is None else int(out_format)
    d = x.shape[-1]
    rows = x.numel() // d
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16 if fmt == LN_OUT_BF16 else torch.float32, device=x.device)
    _check(lib().wenc_layernorm(_ptr(x), _ptr(w), _ptr(b), _ptr(out), rows, d, eps, fmt, _stream(stream)))
    return out


def linear(a, w, bias, epilogue: int = EPI_BIAS_BF16, resid=None, out=None, stream=None):
    """out = epilogue(a w^T + bias); a bf16 [M, K], w bf16 [N, K], bias float32 [N]."""
    import torch
    _require(a, torch.bfloat16, "a")
    _require(w, torch.bfloat16, "w")
    _require(bias, torch.float32, "bias")
    M, K = a.shape
    N = w.shape[0]
    if out is None:
        dt = torch.float32 if epilogue == EPI_BIAS_RESID_F32 else torch.bfloat16
        out = torch.empty((M, N), dtype=dt, device=a.device)
    _check(lib().wenc_linear(_ptr(a), _ptr(w), _ptr(bias), _ptr(resid), _ptr(out), M, N, K, epilogue, _stream(stream)))
    return out


def linear_tf32(a, w, bias, epilogue: int = EPI_BIAS_BF16, resid=None, out=None, stream=None):
    """out = epilogue(a w^T + bias) on TF32 tensor cores; a float32 [M, K], w float32 [N, K].

    Epilogues 0 and 1 write float32 rounded to TF32, epilogue 2 float32 (resid + product).
    """
    import torch
    _require(a, torch.float32, "a")
    _require(w, torch.float32, "w")
    _require(bias, torch.float32, "bias")
    M, K = a.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=a.device)
    _require(out, torch.float32, "out")
    _check(lib().wenc_linear_tf32(_ptr(a), _ptr(w), _ptr(bias), _ptr(resid), _ptr(out), M, N, K, epilogue,
                                  _stream(stream)))
    return out


def attention_tf32(q, k, v, out=None, stream=None):
    """out = softmax(q k^T / 8) v per (window, head) with TF32 products; float32 [B, T, H, 64]."""
    import torch
    for n, t in (("q", q), ("k", k), ("v", v)):
        _require(t, torch.float32, n)
    B, T, H, hd = q.shape
    if out is None:
        out = torch.empty_like(q)
    _require(out, torch.float32, "out")
    _check(lib().wenc_attention_tf32(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, T, H, hd, _stream(stream)))
    return out


def selftest_gemm_pair_abort(a, w, bias, stop_after: int, out=None, stream=None):
    """Launch the CTA-pair GEMM self-test (the odd CTA of each pair stops after `stop_after`
    k-blocks); returns the (undefined) output tensor; read the outcome with sync_status()."""
    import torch
    _require(a, torch.bfloat16, "a")
    _require(w, torch.bfloat16, "w")
    _require(bias, torch.float32, "bias")
    M, K = a.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    _check(lib().wenc_selftest_gemm_pair_abort(_ptr(a), _ptr(w), _ptr(bias), _ptr(out), M, N, K, int(stop_after),
                                              _stream(stream)))
    return out


def selftest_attention_abort(q, k, v, stop_after: int, out=None, stream=None):
    """Launch the attention self-test (its producer stops after `stop_after` K tiles); returns the
    (undefined) output; read the outcome with sync_status()."""
    import torch
    for n, t in (("q", q), ("k", k), ("v", v)):
        _require(t, torch.bfloat16, n)
    B, T, H, hd = q.shape
    if out is None:
        out = torch.empty_like(q)
    _check(lib().wenc_selftest_attention_abort(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, T, H, int(stop_after),
                                              _stream(stream)))
    return out


def selftest_wait_timeout(stream=None):
    """Launch the bounded-wait self-test (returns immediately; read it with sync_status())."""
    _check(lib().wenc_selftest_wait_timeout(_stream(stream)))


def gemm_schedule(M: int, N: int, pair: bool, max_units: int):
    """Host-only replay of a GEMM launch's tile schedule (see wenc_selftest_gemm_schedule).

    Returns (cover, unit_halves, units, halves): cover[t, h] = how often column half h of tile t
    is computed, unit_halves[u] = half tiles computed by unit u (u < units)."""
    import numpy as np
    rows = 256 if pair else 128
    bn = 256 if pair or N % 256 == 0 else 128
    tiles = -(-M // rows) * (N // bn)
    cover = (ctypes.c_int * max(2 * tiles, 2))()
    unit_halves = (ctypes.c_int * max_units)()
    units, halves = ctypes.c_int(), ctypes.c_int()
    _check(lib().wenc_selftest_gemm_schedule(M, N, int(pair), max_units, cover, len(cover), unit_halves,
                                             ctypes.byref(units), ctypes.byref(halves)))
    cov = np.frombuffer(cover, dtype=np.int32, count=2 * tiles).reshape(tiles, 2).copy()
    work = np.frombuffer(unit_halves, dtype=np.int32, count=units.value).copy()
    return cov, work, units.value, halves.value


def sync_status(encoder: Encoder | None = None):
    _check(lib().wenc_sync_status(encoder.handle if encoder is not None else None))
