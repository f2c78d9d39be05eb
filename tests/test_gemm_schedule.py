"""The GEMM's tile schedule, replayed on the host through the code the kernel runs.

wenc_selftest_gemm_schedule sizes a launch exactly as the launchers do and walks every unit's
work items with the kernel's own schedule (no device work). For shapes of every workload and
for edge cases, every column half of every output tile must be computed exactly once, the
units' shares of whole tiles may differ by at most one tile, and a split last wave is used only
where it leaves no more units than the launch has."""
import numpy as np
import pytest

from transformer_encoder_gb300 import WencError, gemm_schedule

# M values: every workload's rows (B x 1500 at B = 1, 2, 4, 8, 16), ragged and tiny cases
MS = [1, 100, 128, 129, 255, 256, 257, 1500, 3000, 6000, 12000, 24000, 48000]
# N values: the block's widths at the five dims (d, 3d, f) and the stem's and cross K/V's
NS = [256, 384, 512, 768, 1152, 1280, 1536, 2048, 2304, 3072, 3840, 5120, 81920]


def _check(M, N, pair, max_units):
    cover, work, units, halves = gemm_schedule(M, N, pair, max_units)
    rows = 256 if pair else 128
    bn = 256 if pair or N % 256 == 0 else 128
    tiles = -(-M // rows) * (N // bn)
    assert cover.shape == (tiles, 2)
    assert (cover == 1).all(), (M, N, pair, max_units)
    assert 1 <= units <= max_units
    assert work.sum() == 2 * tiles
    whole = work // 2  # whole tiles per unit (a half-width unit adds one half)
    assert whole.max() - whole.min() <= 1
    if halves:
        n_tail = tiles % units
        assert 0 < 2 * n_tail <= max_units
        assert ((work % 2) == 1).sum() == 2 * n_tail
    else:
        assert (work % 2 == 0).all()
    return units, halves


@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("max_units", [1, 7, 74, 76, 148, 152])
def test_every_tile_half_is_computed_once(pair, max_units):
    for M in MS:
        for N in NS:
            if pair and N % 256:
                continue
            _check(M, N, pair, max_units)


def test_large_dims_launch_sizes():
    # fc2 / out-projection at B = 16 on CTA pairs: 94 x 5 = 470 tiles on 76 pairs; the 14 left
    # over run as 28 half-width units
    cover, work, units, halves = gemm_schedule(24000, 1280, True, 76)
    assert (units, halves) == (76, 1) and sorted(set(work.tolist())) == [12, 13]
    # one window: 6 x 5 = 30 pair tiles, every one split in two (60 units)
    assert gemm_schedule(1500, 1280, True, 76)[2:] == (60, 1)
    # QKV at B = 16: 94 x 15 = 1410 tiles, 42 left over: too many to split
    assert gemm_schedule(24000, 3840, True, 76)[2:] == (76, 0)
    # single CTAs: 188 x 5 = 940 tiles on 152 SMs, the last 28 split
    assert gemm_schedule(24000, 1280, False, 152)[2:] == (152, 1)


def test_unsupported_shapes_are_refused():
    with pytest.raises(WencError):
        gemm_schedule(100, 384, True, 76)  # pairs need N % 256 == 0
    with pytest.raises(WencError):
        gemm_schedule(100, 200, False, 152)  # N % 128 != 0
    with pytest.raises(WencError):
        gemm_schedule(0, 256, False, 152)
