"""Failure detection on the GPU without a fault: bounded waits run out and are reported.

The self-test kernel waits on an mbarrier that nothing arrives on, with the same bounded
wait every kernel of the library uses. The wait must give up after about a second, record
WENC_ERR_DEVICE_TIMEOUT in the device error word and let the kernel return, leaving the
context usable for the next launch.
"""
import time

import numpy as np
import pytest

import synth
from helpers import attention_gate, bf16_to_f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch
    from transformer_encoder_gb300 import WencError, attention, selftest_wait_timeout, sync_status
    sync_status()  # start from a clear error word
    t0 = time.time()
    selftest_wait_timeout()
    with pytest.raises(WencError, match="DEVICE_TIMEOUT") as ei:
        sync_status()
    elapsed = time.time() - t0
    assert "site 99" in str(ei.value)
    assert 0.5 < elapsed < 30.0
    sync_status()  # the word was cleared by the read
    # the context still runs real work correctly
    q, k, v = synth.make_qkv(1, 300, 2, 64, seed=3)
    to_t = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    out = attention(to_t(q), to_t(k), to_t(v))
    torch.cuda.synchronize()
    f = lambda a: synth.bf16_bits_to_f32(a).reshape(1, 300, 128)
    attention_gate(bf16_to_f64(out).reshape(1, 300, 128), f(q), f(k), f(v), 2, what="after the timeout")
    sync_status()


@pytest.mark.parametrize("stop_after", [0, 3])
def test_cta_pair_gemm_abort_drains_and_context_survives(stop_after):
    """The odd CTA of every pair gives up after `stop_after` k-blocks; the even CTA's waits then
    run out, the pair drains its copies in order and both CTAs exit: the status reads
    DEVICE_TIMEOUT within a few seconds and the same GEMM, run normally next, is correct."""
    import torch

    import oracle
    from transformer_encoder_gb300 import WencError, linear, selftest_gemm_pair_abort, sync_status
    sync_status()
    M, N, K = 1000, 512, 1280  # 4 x 2 pair tiles (fewer than the pairs of a GB300), 20 k-blocks
    rng = np.random.default_rng(31 + stop_after)
    a = synth.round_to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    wt = synth.round_to_bf16((0.05 * rng.standard_normal((N, K))).astype(np.float32))
    bias = (0.1 * rng.standard_normal(N)).astype(np.float32)
    ta = torch.from_numpy(a).cuda().to(torch.bfloat16)
    tw = torch.from_numpy(wt).cuda().to(torch.bfloat16)
    tb = torch.from_numpy(bias).cuda()
    t0 = time.time()
    selftest_gemm_pair_abort(ta, tw, tb, stop_after)
    with pytest.raises(WencError, match="DEVICE_TIMEOUT"):
        sync_status()
    assert time.time() - t0 < 30.0
    sync_status()  # the word was cleared by the read
    out = linear(ta, tw, tb)
    torch.cuda.synchronize()
    ref = oracle.linear(a, wt, bias)
    got = bf16_to_f64(out)
    assert (np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 2e-5 * np.sqrt(np.mean(ref * ref))).all()
    sync_status()


@pytest.mark.parametrize("stop_after", [0, 40])
def test_attention_abort_drains_and_context_survives(stop_after):
    """The attention's TMA producer gives up after `stop_after` K tiles in every CTA (B 16, H 20,
    T 1500: ~156 tiles per CTA, so 40 stops it mid-way through its items). The MMA and softmax
    warps see the abort and stop, the copies in flight drain and TMEM is freed: the status reads
    DEVICE_TIMEOUT within seconds, and attention run normally next passes the oracle gate."""
    import torch
    from transformer_encoder_gb300 import WencError, attention, selftest_attention_abort, sync_status
    sync_status()
    g = torch.Generator(device="cuda").manual_seed(9)
    q, k, v = (torch.randn(16, 1500, 20, 64, device="cuda", generator=g).to(torch.bfloat16) for _ in range(3))
    t0 = time.time()
    selftest_attention_abort(q, k, v, stop_after)
    with pytest.raises(WencError, match="DEVICE_TIMEOUT") as ei:
        sync_status()
    assert time.time() - t0 < 30.0
    assert "site 31" in str(ei.value)
    sync_status()
    del q, k, v
    qs, ks, vs = synth.make_qkv(2, 700, 3, 64, seed=4)
    to_t = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    out = attention(to_t(qs), to_t(ks), to_t(vs))
    torch.cuda.synchronize()
    f = lambda a: synth.bf16_bits_to_f32(a).reshape(2, 700, 192)
    attention_gate(bf16_to_f64(out).reshape(2, 700, 192), f(qs), f(ks), f(vs), 3, what="after the attention abort")
    sync_status()
