"""Pins for the oracle's Philox4x32-10: the published known-answer vectors
(tests/golden/philox4x32_10_kat.txt) and the uniform derived from it."""

import os

import numpy as np
from scipy import stats

from oracle import philox4x32_10, philox_uniform, STREAM_ACCEPT, STREAM_RESAMPLE

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            rows.append([int(w, 16) for w in line.split()])
    return rows


def test_known_answer_vectors():
    rows = _kat()
    assert len(rows) == 3
    for w in rows:
        out = philox4x32_10(*w[:6])
        assert [int(o) for o in out] == w[6:]


def test_vectorised_equals_scalar():
    c = np.arange(50, dtype=np.uint64)
    vec = philox4x32_10(c, 7, 1, 3, 0xDEADBEEF, 0x12345678)
    for i in (0, 13, 49):
        one = philox4x32_10(int(c[i]), 7, 1, 3, 0xDEADBEEF, 0x12345678)
        assert [int(v[i]) for v in vec] == [int(o) for o in one]


def test_uniform_grid_and_distribution():
    n = np.arange(1_000_000)
    u = philox_uniform(0, 0, n, 3, STREAM_ACCEPT)
    assert u.min() >= 0.0 and u.max() < 1.0
    assert np.all(u * 2.0 ** 24 == np.floor(u * 2.0 ** 24))
    assert stats.kstest(u, "uniform").pvalue > 1e-3
    # Streams, positions, offsets and seeds give different draws.
    assert not np.array_equal(u[:1000], philox_uniform(0, 0, n[:1000], 3, STREAM_RESAMPLE))
    assert not np.array_equal(u[:1000], philox_uniform(0, 0, n[:1000], 4, STREAM_ACCEPT))
    assert not np.array_equal(u[:1000], philox_uniform(0, 1, n[:1000], 3, STREAM_ACCEPT))
    assert not np.array_equal(u[:1000], philox_uniform(1 << 32, 0, n[:1000], 3, STREAM_ACCEPT))
