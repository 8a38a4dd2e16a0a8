"""Pins of the oracle's Philox4x32-10 and uniform stream (CPU only)."""
import numpy as np
import pytest
from scipy import stats

import oracle
from conftest import golden


def test_philox_known_answers():
    rows = golden("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for r in rows:
        vals = [int(x, 16) for x in r]
        out = oracle.philox4x32_10(vals[0:4], vals[4:6])
        assert [int(x) for x in out] == vals[6:10]


def test_uniform_mapping_matches_block_function():
    # counter = (b, pos, draw // 4, 0), key = (seed lo, seed hi), word draw % 4, top 24 bits
    seed = 0x0123456789ABCDEF
    for b, pos, draw in [(0, 0, 0), (3, 2, 1), (1000, 15, 3), (7, 1, 5)]:
        out = oracle.philox4x32_10([b, pos, draw // 4, 0], [seed & 0xFFFFFFFF, seed >> 32])
        want = (int(out[draw % 4]) >> 8) / 2.0 ** 24
        assert oracle.uniform(seed, b, pos, draw) == want


def test_uniform_range_and_grid():
    us = np.array([oracle.uniform(5, b, p, d) for b in range(200) for p in range(8) for d in (0, 1)])
    assert us.min() >= 0.0 and us.max() <= 1.0 - 2.0 ** -24
    assert np.all(us * 2 ** 24 == np.floor(us * 2 ** 24))


def test_uniform_is_uniform():
    us = np.array([oracle.uniform(11, b, p, 0) for b in range(4000) for p in range(5)])
    assert stats.kstest(us, "uniform").pvalue > 1e-3
    h, _ = np.histogram(us, bins=32, range=(0, 1))
    assert stats.chisquare(h).pvalue > 1e-3
    # draws 0 and 1 of the same counter are not correlated
    u0 = np.array([oracle.uniform(11, b, 0, 0) for b in range(4000)])
    u1 = np.array([oracle.uniform(11, b, 0, 1) for b in range(4000)])
    assert abs(np.corrcoef(u0, u1)[0, 1]) < 0.06


@pytest.mark.parametrize("seed", [0, 1, 2**32 + 7, 2**64 - 1])
def test_uniform_depends_on_every_key_part(seed):
    a = oracle.uniform(seed, 1, 2, 0)
    assert a != oracle.uniform(seed ^ 1, 1, 2, 0)
    assert a != oracle.uniform(seed ^ (1 << 40), 1, 2, 0)
    assert a != oracle.uniform(seed, 2, 2, 0)
    assert a != oracle.uniform(seed, 1, 3, 0)
    assert a != oracle.uniform(seed, 1, 2, 1)
