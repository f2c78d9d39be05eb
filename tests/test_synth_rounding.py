"""The operand-format roundings of the input generators, checked against their definitions.

round_to_bf16 keeps 8 significant bits (round to nearest, ties to even); round_to_tf32 keeps
11 (10 explicit mantissa bits, round to nearest, ties away from zero). Both are checked by
brute force against the two neighbouring grid points of each input.
"""
import numpy as np

import synth


def _neighbours(x: np.ndarray, drop_bits: int):
    """The grid points just below and above |x| (grid: the low drop_bits bits cleared)."""
    u = np.abs(x).view(np.uint32)
    mask = np.uint32((1 << drop_bits) - 1)
    lo = (u & ~mask).view(np.float32).astype(np.float64)
    hi = ((u & ~mask) + np.uint32(1 << drop_bits)).view(np.float32).astype(np.float64)
    return lo, hi


def _check(rounded, x, drop_bits, ties_away):
    x64 = np.abs(x.astype(np.float64))
    r = np.abs(rounded.astype(np.float64))
    assert (np.signbit(rounded) == np.signbit(x)).all()
    assert ((np.abs(rounded).view(np.uint32) & np.uint32((1 << drop_bits) - 1)) == 0).all()
    lo, hi = _neighbours(x, drop_bits)
    d_lo, d_hi = x64 - lo, hi - x64
    want = np.where(d_lo < d_hi, lo, hi)
    tie = d_lo == d_hi
    if ties_away:
        want = np.where(tie, hi, want)
    else:  # ties to even: the neighbour whose last kept bit is 0
        lo_even = ((np.abs(x).view(np.uint32) >> np.uint32(drop_bits)) & 1) == 0
        want = np.where(tie, np.where(lo_even, lo, hi), want)
    assert (r == want).all()


def _samples():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    # exact ties and near-ties for both grids
    base = rng.standard_normal(2000).astype(np.float32)
    ties = []
    for bits in (13, 16):
        u = base.view(np.uint32) & ~np.uint32((1 << bits) - 1)
        for off in ((1 << (bits - 1)), (1 << (bits - 1)) - 1, (1 << (bits - 1)) + 1):
            ties.append((u + np.uint32(off)).view(np.float32))
    return np.concatenate([x, *ties, np.float32([0.0, -0.0, 1.0, -1.0])])


def test_round_to_tf32_is_nearest_ties_away():
    x = _samples()
    _check(synth.round_to_tf32(x), x, 13, ties_away=True)


def test_round_to_bf16_is_nearest_ties_even():
    x = _samples()
    _check(synth.round_to_bf16(x), x, 16, ties_away=False)


def test_tf32_grid_values():
    x = np.float32([1.0, 1 + 2 ** -11, 1 + 3 * 2 ** -11, -(1 + 2 ** -11), 1 + 2 ** -12, 2 ** -10])
    want = np.float32([1.0, 1 + 2 ** -10, 1 + 2 ** -9, -(1 + 2 ** -10), 1.0, 2 ** -10])
    assert (synth.round_to_tf32(x) == want).all()
