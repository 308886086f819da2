"""Pins the oracle's Philox4x64-10 to numpy's independent implementation.

numpy.random.Philox is a Philox-4x64 generator with 10 rounds.  Its bit
generator advances the 256-bit counter before producing each block, so a
generator created with counter c - 1 emits the block of counter c first.
"""

import numpy as np
import pytest

from oracle import philox

M64 = (1 << 64) - 1


def numpy_block(key_words, counter_words):
    key = key_words[0] | (key_words[1] << 64)
    ctr = sum(w << (64 * i) for i, w in enumerate(counter_words))
    gen = np.random.Philox(key=key, counter=(ctr - 1) % (1 << 256))
    return tuple(int(gen.random_raw()) for _ in range(4))


CASES = [
    ((0, 0), (0, 0, 0, 0)),
    ((0, 0), (1, 0, 0, 0)),
    ((1, 0), (0, 0, 0, 0)),
    ((12345, 0), (7, 3, 2, 0)),
    ((M64, M64), (M64, M64, M64, M64)),
    ((0xDEADBEEF, 0x1234), (1 << 63, 99, 4, 1)),
]


@pytest.mark.parametrize("key,ctr", CASES)
def test_block_matches_numpy(key, ctr):
    assert philox.philox4x64_10(ctr, key) == numpy_block(key, ctr)


def test_random_blocks_match_numpy():
    rng = np.random.default_rng(7)
    for _ in range(200):
        key = tuple(int(x) for x in rng.integers(0, 1 << 64, size=2, dtype=np.uint64))
        ctr = tuple(int(x) for x in rng.integers(0, 1 << 64, size=4, dtype=np.uint64))
        assert philox.philox4x64_10(ctr, key) == numpy_block(key, ctr)


def test_uniform_layout():
    # key = (seed, 0), counter = (offset, row, draw, 0), u = top 53 bits of word 0
    seed, offset, row, draw = 5, 11, 3, 2
    w0 = numpy_block((seed, 0), (offset, row, draw, 0))[0]
    u = philox.uniform(seed, offset, row, draw)
    assert u == (w0 >> 11) * 2.0 ** -53
    assert 0.0 <= u < 1.0


def test_uniforms_are_uniform():
    us = np.array([philox.uniform(0, 0, r, 0) for r in range(20000)])
    hist, _ = np.histogram(us, bins=20, range=(0.0, 1.0))
    expected = us.size / 20
    chi2 = float(np.sum((hist - expected) ** 2 / expected))
    # 19 degrees of freedom: the 0.999 quantile is 43.8
    assert chi2 < 43.8
    assert len(set(us.tolist())) == us.size
