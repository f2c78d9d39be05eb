"""wenc_attention_static: attention for callers that must not allocate device memory.

Some programs that call this library are not allowed to allocate GPU memory while they run:
a host that lends out memory only from its own fixed pool, a serving runtime that forbids
allocation after start-up, or code for which the device synchronisation of an allocation is
too costly. wenc_attention_static gives them split-key attention whose partial results sit in
a static buffer that is part of the library itself. This file checks, through the C ABI, that
its output agrees with wenc_attention (the entry point that needs no scratch at all) within the
attention tolerance of the other tests, on two calls in a row with different shapes, that a
repeated call gives the same bits (the buffer's leftover contents do not matter), that free
device memory does not move, and that a problem too large for the buffer is refused.

It sits in a file of its own that pytest collects last, so a run that stops at the first
failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest

import synth
from helpers import attention_gate, bf16_to_f64

pytestmark = pytest.mark.gpu


def _case(B, T, H, seed):
    import torch
    q, k, v = synth.make_qkv(B, T, H, 64, seed=seed)
    to_t = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    to_f = lambda a: synth.bf16_bits_to_f32(a).reshape(B, T, H * 64)
    return (to_t(q), to_t(k), to_t(v)), (to_f(q), to_f(k), to_f(v))


def _static_call(L, tq, tk, tv, out, B, T, H):
    import torch
    vp = ctypes.c_void_p
    stream = vp(torch.cuda.current_stream().cuda_stream)
    return L.wenc_attention_static(vp(tq.data_ptr()), vp(tk.data_ptr()), vp(tv.data_ptr()), vp(out.data_ptr()), B, T,
                                   H, 64, stream)


def _check_against_existing(got, ref_existing, q, k, v, H, what):
    import oracle
    attention_gate(got, q, k, v, H, what=what)
    # both outputs lie within the bf16 rounding bound of the exact result, so within twice it
    # of each other
    ref = oracle.attention(q, k, v, H)
    absv = oracle.attention(q, k, np.abs(np.asarray(v, np.float64)), H)
    bound = 2 * 1.1 * 2.0 ** -9 * (np.abs(ref) + absv) + 2e-6
    assert (np.abs(got - ref_existing) <= bound).all(), what


def test_static_scratch_attention_matches_wenc_attention():
    import torch
    from transformer_encoder_gb300 import attention, lib, sync_status
    L = lib()
    shapes = [(1, 1500, 6, 11), (2, 700, 3, 12)]  # tiny-model heads; a ragged 700-key window
    first = None
    for B, T, H, seed in shapes:
        (tq, tk, tv), (q, k, v) = _case(B, T, H, seed)
        out = torch.empty_like(tq)
        assert _static_call(L, tq, tk, tv, out, B, T, H) == 0, L.wenc_last_error()
        existing = attention(tq, tk, tv)
        torch.cuda.synchronize()
        sync_status()
        got = bf16_to_f64(out).reshape(B, T, H * 64)
        _check_against_existing(got, bf16_to_f64(existing).reshape(B, T, H * 64), q, k, v, H,
                                what=f"static-scratch attention B={B} T={T} H={H}")
        if first is None:
            first = (tq, tk, tv, out.clone(), B, T, H)
    # the first shape again, after the second call overwrote the buffer: identical bits, and no
    # device memory taken by the call
    tq, tk, tv, out_first, B, T, H = first
    again = torch.empty_like(out_first)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    assert _static_call(L, tq, tk, tv, again, B, T, H) == 0, L.wenc_last_error()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert torch.equal(again.view(torch.int16), out_first.view(torch.int16))


def test_static_scratch_attention_refuses_oversized_problems():
    import torch
    from transformer_encoder_gb300 import lib
    L = lib()
    cap = L.wenc_attention_static_capacity()
    assert cap == 16 << 20
    # B*H*T large enough that even two splits need more than the buffer
    B, T, H = 64, 1500, 20
    buf = torch.empty(16, dtype=torch.bfloat16, device="cuda")  # never read: the call is refused first
    vp = ctypes.c_void_p
    st = L.wenc_attention_static(vp(buf.data_ptr()), vp(buf.data_ptr()), vp(buf.data_ptr()), vp(buf.data_ptr()), B, T,
                                 H, 64, vp(torch.cuda.current_stream().cuda_stream))
    assert st == 1
    assert b"static buffer" in L.wenc_last_error()
    # a following call that succeeds clears that message
    (q, k, v), _ = _case(1, 300, 2, 5)
    small = torch.empty_like(q)
    assert _static_call(L, q, k, v, small, 1, 300, 2) == 0
    torch.cuda.synchronize()
    assert L.wenc_last_error() == b""
