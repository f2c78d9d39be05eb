"""Child process of test_gpu_gemm_forms: runs a fixed set of GEMMs and one large-dims forward
and saves the outputs to an .npz file. The GEMM form (CTA pairs or single CTAs) is chosen by the
WENC_GEMM_PAIR environment variable, which the library reads once per process, so each form
runs in a process of its own."""
import sys

import numpy as np
import torch

import synth
from helpers import make_encoder

# (M, N, K, epilogue): 256-column tiles with a ragged last row block, a partial last wave and
# a single tile
LINEAR_CASES = [(1537, 2048, 512, 1), (3000, 1280, 1280, 2), (129, 256, 64, 0), (1500, 1280, 5120, 2),
                (2900, 3840, 1280, 0)]


def linear_case(M, N, K, epi):
    from transformer_encoder_gb300 import linear
    rng = np.random.default_rng(1000 + M + N + K + epi)
    a = synth.round_to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    wt = synth.round_to_bf16((0.05 * rng.standard_normal((N, K))).astype(np.float32))
    bias = (0.1 * rng.standard_normal(N)).astype(np.float32)
    resid = rng.standard_normal((M, N)).astype(np.float32) if epi == 2 else None
    out = linear(torch.from_numpy(a).cuda().to(torch.bfloat16), torch.from_numpy(wt).cuda().to(torch.bfloat16),
                 torch.from_numpy(bias).cuda(), epi, resid=torch.from_numpy(resid).cuda() if resid is not None else None)
    torch.cuda.synchronize()
    return (out.view(torch.int16) if out.dtype == torch.bfloat16 else out).cpu().numpy()


def main(path):
    res = {f"linear_{M}_{N}_{K}_{e}": linear_case(M, N, K, e) for M, N, K, e in LINEAR_CASES}
    w = synth.WORKLOADS["large_pair"]
    enc, _, _, rng = make_encoder(w, keep_host_layers=False, max_batch=2)
    x = synth.make_input(w, rng)[:2]
    y = enc.forward(torch.from_numpy(np.ascontiguousarray(x)).cuda())
    torch.cuda.synchronize()
    enc.sync_status()
    res["forward_large_pair_b2"] = y.cpu().numpy()
    np.savez(path, **res)


if __name__ == "__main__":
    main(sys.argv[1])
