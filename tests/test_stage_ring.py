"""The page ring's lap arithmetic, on the CPU.

The tensor-core decode kernel puts page k of a CTA's slice in stage k mod n of a ring of n stages
(any n from 2 to 16, as many as fit in shared memory) and takes the lap k / n as the high 32 bits
of k * ceil(2^32 / n).  That quotient is exact for every k below 2^32 / n, so for every page index a
slice can hold (below 2^28).  Checked here for every k below 2^22 and at the top of the range.
"""
import numpy as np


def lap(k, n):
    magic = np.uint64((2**32 + n - 1) // n)
    return (k.astype(np.uint64) * magic) >> np.uint64(32)


def test_multiply_high_lap_is_the_quotient():
    dense = np.arange(0, 1 << 22, dtype=np.uint64)
    top = np.arange((1 << 28) - (1 << 16), 1 << 28, dtype=np.uint64)
    for n in range(2, 17):
        for k in (dense, top):
            q = lap(k, n)
            assert np.array_equal(q, k // np.uint64(n)), n
            assert ((2**32 + n - 1) // n) < 2**32  # the constant fits the kernel's 32-bit operand


def test_one_stage_constant_would_not_fit():
    # why the launcher refuses a ring of one stage: ceil(2^32 / 1) needs 33 bits
    assert (2**32 + 1 - 1) // 1 == 2**32
