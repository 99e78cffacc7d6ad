"""The range of bf16 values whose squares the norm kernels treat as exact, checked against exact
arithmetic over every bf16 bit pattern (no GPU).

The norm kernels keep sums of squares as float pairs, adding each square's FMA residual.  For a bf16
value whose magnitude bits (exponent field << 7 | mantissa) lie in [kExactSquareMin, kExactSquareMax],
or that is zero, the fp32 square is exact, so the residual is +0 and the kernels leave it out.  The
constants are read from the kernel header; float64 holds every such square exactly (at most 16
significant bits), so "exact in fp32" is "converting the float64 square to float32 and back changes
nothing, and the result is finite".
"""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _constants():
    src = open(os.path.join(ROOT, "zero_sharded_mixed_local_gb300", "csrc", "pair_sum.cuh")).read()
    lo = int(re.search(r"kExactSquareMin\s*=\s*(0x[0-9A-Fa-f]+)u", src).group(1), 16)
    hi = int(re.search(r"kExactSquareMax\s*=\s*(0x[0-9A-Fa-f]+)u", src).group(1), 16)
    return lo, hi


def _square_is_fp32(bits):
    x = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    sq = x * x
    with np.errstate(over="ignore", invalid="ignore"):
        r = sq.astype(np.float32)
    return np.isfinite(r) & (r.astype(np.float64) == sq)


def test_every_value_in_the_range_squares_exactly():
    lo, hi = _constants()
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mag = bits & 0x7FFF
    in_range = ((mag >= lo) & (mag <= hi)) | (mag == 0)
    assert in_range.sum() == 2 * (hi - lo + 1) + 2  # both signs, and +0 / -0
    assert _square_is_fp32(bits[in_range]).all()


def test_the_range_ends_where_squares_stop_being_exact():
    lo, hi = _constants()
    # one below: exponent field 59 with an odd mantissa, whose square needs a bit at 2^-150
    assert not _square_is_fp32(np.array([lo - 1, 0x8000 | (lo - 1)], np.uint16)).any()
    # one above: 2^64, whose square 2^128 overflows fp32
    assert not _square_is_fp32(np.array([hi + 1, 0x8000 | (hi + 1)], np.uint16)).any()
    # the ends themselves are the exponent fields 60 and 190
    assert lo >> 7 == 60 and lo & 0x7F == 0 and hi >> 7 == 190 and hi & 0x7F == 0x7F


def test_bf16_subnormals_infinities_and_nan_lie_outside_the_range():
    lo, hi = _constants()
    special = np.array([0x0001, 0x007F, 0x7F80, 0x7FC0, 0xFF80], np.uint16)
    assert (((special & 0x7FFF) < lo) | ((special & 0x7FFF) > hi)).all()
    assert not _square_is_fp32(special).any()
