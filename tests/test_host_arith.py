"""Integer arithmetic the planner's schedule stage relies on.

The schedule stage divides task indices by divisors fixed for the whole
launch (padded rows, Q tile rows per sample, the GQA group) with one
multiply and a shift: m = ceil(2^(31+L) / d), L = ceil(log2 d), quotient
floor(x m / 2^(31+L)) for 0 <= x < 2^31 ("Division by Invariant Integers
using Multiplication", Granlund and Montgomery, 1994).  These checks pin
the two facts the kernel needs: m fits in 32 bits for every divisor below
2^31, and the quotient is exact (checked exhaustively where that is cheap,
else at the edges of every quotient bucket and at random points)."""
import random

import pytest


def multiplier(d):
    L = 0
    while (1 << L) < d:
        L += 1
    return -(-(1 << (31 + L)) // d), 31 + L


def quotient(x, d):
    m, sh = multiplier(d)
    return (x * m) >> sh


@pytest.mark.parametrize("d", [1, 2, 3, 7, 64, 127, 128, 129, 255, 256, 257, 1000, 4095, 65537,
                               (1 << 20) + 3, (1 << 30) - 1, 1 << 30, (1 << 30) + 1, (1 << 31) - 1])
def test_multiplier_fits_and_quotients_exact(d):
    m, sh = multiplier(d)
    assert 0 < m < (1 << 32)
    assert (1 << sh) <= m * d <= (1 << sh) + (1 << (sh - 31))  # the method's error bound
    rng = random.Random(d)
    xs = {0, 1, d - 1, d, d + 1, (1 << 31) - 1, (1 << 31) - 2}
    for q in (1, 2, 3, 1000, ((1 << 31) - 1) // d):
        for r in (-1, 0, 1):
            x = q * d + r
            if 0 <= x < (1 << 31):
                xs.add(x)
    xs.update(rng.randrange(1 << 31) for _ in range(2000))
    for x in xs:
        assert quotient(x, d) == x // d, (x, d)


def test_small_divisors_exhaustive_below_2_pow_16():
    for d in range(1, 300):
        for x in range(0, 1 << 16, 7):
            assert quotient(x, d) == x // d, (x, d)
