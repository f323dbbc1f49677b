"""The reciprocal division of the kernels' ring and tile indices (SmallDiv in csrc/common.cuh):
q / d as the high 32 bits of q * m with m = floor((2^32 - 1) / d) + 1, d = 1 passed through. The
kernels rely on it being exact for every q below 2^32 / (d - 1); the separate-path kernel falls
back to a hardware division at and beyond floor((2^32 - 1) / (rbpg - 1)) (capped at 2^31 - 1).
Checked here with Python integers, exhaustively for small q and at the bound for every divisor
the kernels can see (ring depths, chunks per row, row blocks per group, warp sets)."""
import numpy as np


def recip(d):
    return (0xFFFFFFFF // d + 1) if d > 1 else 0


def small_div(q, d):
    return (q * recip(d)) >> 32 if d > 1 else q


def qlim(d):
    """First index the kernels no longer divide by the reciprocal (the separate-path bound)."""
    return min(0xFFFFFFFF // (d - 1), 0x7FFFFFFF) if d > 1 else 0x7FFFFFFF


def test_exhaustive_small_indices():
    q = np.arange(0, 1 << 16, dtype=np.uint64)
    for d in range(1, 1025):
        m = np.uint64(recip(d))
        got = (q * m) >> np.uint64(32) if d > 1 else q
        assert np.array_equal(got, q // np.uint64(d)), d


def test_exact_up_to_the_bound():
    rng = np.random.default_rng(7)
    for d in list(range(2, 4097)) + [5000, 12345, 65535, 65536, 1 << 20]:
        lim = qlim(d)
        # the largest indices still divided by the reciprocal, and a random sample below them
        qs = [lim - 1, lim - 2, lim - d, lim - d - 1] + [int(v) for v in rng.integers(0, lim, 64)]
        for q in qs:
            if q >= 0:
                assert small_div(q, d) == q // d, (d, q)
                assert q - small_div(q, d) * d == q % d


def test_power_of_two_divisors_are_exact_everywhere():
    for k in range(1, 31):
        d = 1 << k
        for q in (0, 1, d - 1, d, 0x7FFFFFFF, 0xFFFFFFFF):
            assert small_div(q, d) == q // d


def test_divisor_one_passes_through():
    for q in (0, 1, 12345, 0x7FFFFFFF):
        assert small_div(q, 1) == q
