"""The C ABI without a GPU: libwenc.so builds, loads, exports exactly what include/wenc.h
declares, and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from transformer_encoder_gb300 import lib, lib_path
    from transformer_encoder_gb300.build import build
    build()
    assert os.path.exists(lib_path)
    return lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "wenc.h")).read()
    return sorted(set(re.findall(r"WENC_API\s+[\w\s\*]+?\b(wenc_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("wenc_create", "wenc_forward", "wenc_attention", "wenc_sync_status", "wenc_destroy",
                     "wenc_last_error"):
        assert required in names


def test_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_binding_lists_the_declared_symbols():
    from transformer_encoder_gb300 import EXPORTED_SYMBOLS
    assert sorted(EXPORTED_SYMBOLS) == _declared()


def test_only_declared_symbols_are_exported(L):
    import subprocess
    from transformer_encoder_gb300 import lib_path
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True).stdout
    wenc_syms = sorted({line.split()[-1] for line in out.splitlines() if line.split()[-1].startswith("wenc_")})
    assert wenc_syms == _declared()


def test_version(L):
    assert L.wenc_version().decode().startswith("wenc ")


def test_host_side_argument_errors(L):
    from transformer_encoder_gb300.wenc import Config
    out = ctypes.c_void_p(123)
    assert L.wenc_create(None, None, None, None, None, ctypes.byref(out)) == 1
    assert out.value is None
    assert b"config" in L.wenc_last_error()
    cfg = Config(1, 384, 6, 32, 1536, 1500, 1, 0, 1e-5, 0, 0)  # d != H * hd
    assert L.wenc_create(ctypes.byref(cfg), None, None, None, None, ctypes.byref(out)) == 1
    cfg = Config(1, 384, 12, 32, 1536, 1500, 1, 0, 1e-5, 0, 0)  # hd = 32
    assert L.wenc_create(ctypes.byref(cfg), None, None, None, None, ctypes.byref(out)) == 2
    cfg = Config(1, 384, 6, 64, 1500, 1500, 1, 0, 1e-5, 0, 0)   # ffn not a multiple of 128
    assert L.wenc_create(ctypes.byref(cfg), None, None, None, None, ctypes.byref(out)) == 2
    assert L.wenc_forward(None, None, None, 1, None) == 1
    assert L.wenc_forward_launches(None, 0, 1, 1) == -1
    p = ctypes.c_void_p(256)
    assert L.wenc_attention(p, p, p, p, 1, 10, 2, 32, None) == 2   # hd != 64
    assert L.wenc_attention(p, p, p, p, 0, 10, 2, 64, None) == 1   # B < 1
    assert L.wenc_attention(None, p, p, p, 1, 10, 2, 64, None) == 1
    assert L.wenc_layernorm(p, p, p, p, 10, 100, 1e-5, 1, None) == 2  # d not a multiple of 128
    assert L.wenc_linear(p, p, p, None, p, 10, 128, 64, 2, None) == 1  # residual epilogue without resid
    assert L.wenc_linear(p, p, p, None, p, 10, 100, 64, 0, None) == 2  # N not a multiple of 128
    L.wenc_destroy(None)


def test_host_side_argument_errors_tf32(L):
    from transformer_encoder_gb300.wenc import Config, PREC_TF32
    out = ctypes.c_void_p(123)
    cfg = Config(1, 384, 6, 64, 1536, 1500, 1, 0, 1e-5, 0, 7)  # unknown precision
    assert L.wenc_create(ctypes.byref(cfg), None, None, None, None, ctypes.byref(out)) == 2
    assert b"precision" in L.wenc_last_error()
    cfg = Config(1, 384, 6, 64, 1536, 1500, 1, 0, 1e-5, 0, PREC_TF32)  # valid config, no layers
    assert L.wenc_create(ctypes.byref(cfg), None, None, None, None, ctypes.byref(out)) == 1
    assert b"layers" in L.wenc_last_error()
    p = ctypes.c_void_p(256)
    assert L.wenc_linear_tf32(p, p, p, None, p, 10, 128, 48, 0, None) == 2   # K not a multiple of 32
    assert L.wenc_linear_tf32(p, p, p, None, p, 10, 128, 64, 2, None) == 1   # residual epilogue without resid
    assert L.wenc_linear_tf32(p, p, p, None, p, 10, 128, 64, 3, None) == 1   # unknown epilogue
    assert L.wenc_linear_tf32(p, p, p, None, p, 0, 128, 64, 0, None) == 1    # M < 1
    assert L.wenc_attention_tf32(p, p, p, p, 1, 10, 2, 32, None) == 2       # hd != 64
    assert L.wenc_attention_tf32(p, p, p, p, 1, 0, 2, 64, None) == 1        # T < 1
    assert L.wenc_attention_tf32(p, p, None, p, 1, 10, 2, 64, None) == 1
    assert L.wenc_layernorm(p, p, p, p, 10, 128, 1e-5, 3, None) == 1         # unknown output format


def test_host_side_argument_errors_stem(L):
    from transformer_encoder_gb300.wenc import StemWeights
    p = ctypes.c_void_p(256)
    w = StemWeights(80, 256, 256, 256, 256, 256)
    assert L.wenc_set_stem(None, ctypes.byref(w), None) == 1
    assert b"handle" in L.wenc_last_error()
    assert L.wenc_stem(None, p, p, 1, None) == 1
    assert L.wenc_encode(None, p, p, 1, None) == 1
    assert L.wenc_encode_launches(None) == -1
    assert L.wenc_set_cross_kv(None, 1, None, None, None, None) == 1
    assert L.wenc_cross_kv(None, p, p, 1, None) == 1
