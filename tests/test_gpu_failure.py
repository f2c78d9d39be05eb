"""Failure detection on the GPU without a fault: a bounded wait runs out and is reported.

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
