"""Pins of the oracle's Philox4x32-10 and of the uniform streams."""
import os

import numpy as np
import pytest

from oracle import philox

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat():
    rows = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        rows.append([int(v, 16) for v in line.split()])
    return rows


@pytest.mark.parametrize("row", _kat())
def test_known_answer_vectors(row):
    out = philox.philox4x32_10(*row[:6])
    assert [int(v) for v in out] == row[6:]


def test_uniform_map_is_exact_in_fp32_and_open_interval():
    x = np.array([0, 1, 511, 512, 0xFFFFFFFF, 0x80000000], dtype=np.uint64)
    u = philox.bits_to_uniform(x)
    assert np.all(u > 0) and np.all(u < 1)
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    assert u[0] == 2.0 ** -24 and u[4] == 1 - 2.0 ** -24


def test_streams_are_uniform_and_distinct():
    acc = philox.accept_uniforms(seed=7, offset=3, B=64, R=512).ravel()
    race = philox.race_uniforms(seed=7, offset=3, b=5, V=32768)
    for u in (acc, race):
        hist, _ = np.histogram(u, bins=16, range=(0, 1))
        exp = len(u) / 16
        chi2 = ((hist - exp) ** 2 / exp).sum()
        assert chi2 < 45.0  # chi-square(15) upper tail ~1e-4
    # different offset or seed -> different draws
    assert not np.array_equal(philox.accept_uniforms(7, 4, 2, 8), philox.accept_uniforms(7, 3, 2, 8))
    assert not np.array_equal(philox.accept_uniforms(8, 3, 2, 8), philox.accept_uniforms(7, 3, 2, 8))


def test_race_stream_word_selection():
    # id y uses word (y & 3) of the block for counter y >> 2
    u = philox.race_uniforms(seed=0x1234_5678_9ABC, offset=0, b=2, V=8)
    w = philox.philox4x32_10(1, 2, 1, 0, 0x5678_9ABC, 0x1234)
    assert u[4:8].tolist() == [philox.bits_to_uniform(v) for v in w]
