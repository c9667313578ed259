"""Pins of the oracle's counter-based generator (Philox4x32-10), its uniform
map and its Gumbel variates, against published known answers and distribution
tests.  CPU only."""
import math
import os

import numpy as np
import pytest
from scipy import stats

import oracle


def _kat(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "philox4x32_10_kat.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            w = [int(t, 16) for t in line.split()]
            rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


def test_philox_known_answers(golden_dir):
    rows = _kat(golden_dir)
    assert len(rows) == 3
    for ctr, key, want in rows:
        assert oracle.philox4x32_10(ctr, key) == want


def test_stream_layout_words():
    # counter = (v>>2, k, req, round<<3 | stream), key = (seed lo, seed hi), word v&3
    seed, rnd, stream, req, k = 0x1234567890ABCDEF, 5, 2, 7, 3
    for v in range(0, 12):
        full = oracle.philox4x32_10([v >> 2, k, req, (rnd << 3) | stream],
                                    [seed & 0xffffffff, seed >> 32])
        assert oracle.rng_word(seed, rnd, stream, req, k, v) == full[v & 3]


def test_u01_grid_and_range():
    assert oracle.u01(0) == 2.0 ** -24
    assert oracle.u01(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert oracle.u01(0x1FF) == 2.0 ** -24  # low 9 bits are dropped
    for w in [0, 1 << 9, 12345 << 9, 0xFFFFFE00]:
        m = w >> 9
        assert oracle.u01(w) == (2 * m + 1) / 2.0 ** 24
        # exactly representable in float32
        assert float(np.float32(oracle.u01(w))) == oracle.u01(w)


def test_uniformity_ks_and_streams():
    n = 40000
    u = np.array([oracle.u01(oracle.rng_word(7, 0, 0, 3, 1, v)) for v in range(n)])
    assert stats.kstest(u, "uniform").pvalue > 1e-3
    # a different stream, request, position or round gives an unrelated sequence
    for args in [(7, 0, 1, 3, 1), (7, 0, 0, 4, 1), (7, 0, 0, 3, 2), (7, 1, 0, 3, 1), (8, 0, 0, 3, 1)]:
        u2 = np.array([oracle.u01(oracle.rng_word(*args, v)) for v in range(4000)])
        assert abs(np.corrcoef(u[:4000], u2)[0, 1]) < 0.06
        assert not np.array_equal(u[:4000], u2)


def test_gumbel_distribution():
    # the block noise G = -log(-log u) with u from a word's top 23 bits:
    # CDF exp(-exp(-g)), mean = Euler-Mascheroni, var = pi^2/6
    n = 40000
    g = np.array([oracle.gumbel_from_bits(oracle.rng_word(11, 2, 0, 0, 1, v) >> 9) for v in range(n)])
    assert stats.kstest(g, stats.gumbel_r.cdf).pvalue > 1e-3
    assert abs(g.mean() - 0.5772156649) < 0.03
    assert abs(g.var() - math.pi ** 2 / 6) < 0.06
    # bounded support from the 23-bit grid
    gmax = -math.log(-math.log(1.0 - 2.0 ** -24))
    gmin = -math.log(-math.log(2.0 ** -24))
    assert g.max() <= gmax and g.min() >= gmin
    assert oracle.gumbel_from_bits((1 << 23) - 1) == pytest.approx(gmax, rel=0, abs=1e-12)
