"""Pins of the oracle's randomness: Philox4x32-10 against the published
known-answer vectors, and the (0,1) mapping against its closed form."""
import os

import numpy as np

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat():
    rows = []
    for line in open(GOLD):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(x, 16) for x in line.split()]
        rows.append((w[:4], w[4:6], tuple(w[6:])))
    return rows


def test_philox_known_answers():
    rows = _kat()
    assert len(rows) == 3
    for ctr, key, out in rows:
        assert O.philox4x32_10(ctr, key) == out


def test_counter_packing_and_word_select():
    # counter = (n // 4, i, j, purpose); key = (lo32 seed, hi32 seed); word n % 4
    seed = 0x0123456789ABCDEF
    for (j, i, p, n) in [(0, 1, 1, 0), (5, 3, 2, 7), (511, 16, 4, 148), (3, 9, 3, 2)]:
        blk = O.philox4x32_10([n // 4, i, j, p], [seed & 0xFFFFFFFF, seed >> 32])
        assert O.philox_word(seed, j, i, p, n) == blk[n % 4]


def test_uniform_mapping_closed_form():
    seed = 7
    for n in range(64):
        x = O.philox_word(seed, 2, 3, 1, n)
        u = O.uniform(seed, 2, 3, 1, n)
        assert u == ((x >> 9) + 0.5) / 2 ** 23
        assert 0.0 < u < 1.0
        assert float(np.float32(u)) == u  # exact in fp32


def test_uniform_is_uniform():
    # Kolmogorov-Smirnov on 20000 draws across counters
    from scipy import stats

    us = np.array([O.uniform(11, j, 1, 1, 0) for j in range(20000)])
    assert stats.kstest(us, "uniform").pvalue > 1e-3
    assert us.min() >= 2.0 ** -24 and us.max() <= 1 - 2.0 ** -24
