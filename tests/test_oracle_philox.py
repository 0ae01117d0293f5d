"""Pins of the oracle's random-number layer.

Philox-4x32-10 is pinned to the published known-answer vectors (Salmon et al.,
SC'11; tests/golden/philox4x32_10_kat.txt).  The word-to-uniform map
u = ((w >> 9) + 1/2) 2^-23 is pinned by its extreme values, by exactness in
fp32, and by the moments and a Kolmogorov-Smirnov test of many draws.
"""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        vals = [int(t, 16) for t in line.split()]
        rows.append((vals[0:4], vals[4:6], vals[6:10]))
    return rows


@pytest.mark.parametrize("ctr,key,expect", _kat())
def test_philox_known_answers(orc, ctr, key, expect):
    out = orc.philox4x32_10(ctr, key)
    assert [int(v) for v in out] == expect


def test_philox_word_layout(orc):
    # the helper places (w0, w1, request, cycle<<2 | stream) and the key halves
    seed = 0x0123456789ABCDEF
    ctr = [17, 3, 9, (5 << 2) | 2]
    key = [seed & 0xFFFFFFFF, seed >> 32]
    out = orc.philox4x32_10(ctr, key)
    for lane in range(4):
        assert orc.philox_word(seed, 17, 3, 9, 5, 2, lane) == int(out[lane])


def test_uniform_extremes_and_exactness(orc):
    assert orc.uniform(0) == 2.0 ** -24
    assert orc.uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert orc.uniform(0x1FF) == orc.uniform(0)  # the low 9 bits are dropped
    for w in [0, 1 << 9, 0x80000000, 0xFFFFFFFF, 0xDEADBEEF]:
        u = orc.uniform(w)
        assert 0.0 < u < 1.0
        assert float(np.float32(u)) == u  # exact in binary32: both sides agree bit for bit


def test_uniform_distribution(orc):
    from scipy import stats
    n = 200_000
    words = [orc.philox_word(7, i // 4, 0, 0, 0, 3, i % 4) for i in range(n)]
    u = np.array([orc.uniform(w) for w in words])
    assert abs(u.mean() - 0.5) < 5 * np.sqrt(1 / 12 / n)
    assert abs(u.var() - 1 / 12) < 0.002
    assert stats.kstest(u, "uniform").pvalue > 1e-4
