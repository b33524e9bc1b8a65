"""Pins of the oracle's Philox-4x32-10 copy and its uniform mapping."""

import os

import numpy as np
from scipy import stats

from oracle.philox import philox4x32_10, uniform, PURPOSE_ACCEPT, PURPOSE_RESAMPLE

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kat():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            rows.append([int(v, 16) for v in line.split()])
    return rows


def test_known_answer_vectors():
    kat = _kat()
    assert len(kat) == 3
    for row in kat:
        out = philox4x32_10(*row[:6])
        assert [int(v) for v in out] == row[6:]


def test_vectorised_matches_scalar():
    rng = np.random.default_rng(1)
    c = rng.integers(0, 2**32, size=(4, 257), dtype=np.uint64)
    k = rng.integers(0, 2**32, size=2, dtype=np.uint64)
    vec = philox4x32_10(c[0], c[1], c[2], c[3], k[0], k[1])
    for j in (0, 17, 256):
        one = philox4x32_10(c[0, j], c[1, j], c[2, j], c[3, j], k[0], k[1])
        assert [int(v[j]) for v in vec] == [int(v) for v in one]


def test_uniform_is_exact_dyadic_in_open_interval():
    u = uniform(12345, np.arange(100000, dtype=np.uint64), 3, PURPOSE_ACCEPT)
    assert np.all(u > 0) and np.all(u < 1)
    scaled = u * 2.0**23 - 0.5
    assert np.all(scaled == np.round(scaled))
    assert np.all(np.float32(u) == u)  # exact in fp32 as well


def test_uniform_chi_square():
    u = uniform(7, np.arange(200000, dtype=np.uint64), 0, PURPOSE_RESAMPLE)
    counts = np.bincount((u * 64).astype(int), minlength=64)
    _, pval = stats.chisquare(counts)
    assert pval > 1e-4


def test_counter_fields_separate_streams():
    rows = np.arange(1000, dtype=np.uint64)
    a = uniform(0, rows, 0, PURPOSE_ACCEPT)
    assert not np.array_equal(a, uniform(0, rows, 1, PURPOSE_ACCEPT))
    assert not np.array_equal(a, uniform(0, rows, 0, PURPOSE_RESAMPLE))
    assert not np.array_equal(a, uniform(1, rows, 0, PURPOSE_ACCEPT))
    big = uniform(0, rows + np.uint64(2**32), 0, PURPOSE_ACCEPT)  # row's high word is used
    assert not np.array_equal(a, big)
