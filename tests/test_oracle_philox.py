"""Pins of the oracle's Philox4x32-10.

Known-answer vectors: the Random123 release that accompanies Salmon et al.,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), publishes outputs of
philox4x32 with 10 rounds for three (counter, key) inputs; they are restated
here as test data.
"""
import numpy as np
import pytest

from oracle.philox import bitrev16, pair_draws16, philox4x32

KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF, 0xFFFFFFFF), (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,want", KAT)
def test_known_answer_vectors(ctr, key, want):
    out = philox4x32(np.array(ctr, dtype=np.uint64), key)
    assert tuple(int(x) for x in out) == want


def test_vectorised_equals_scalar():
    rng = np.random.default_rng(0)
    ctr = rng.integers(0, 2 ** 32, size=(64, 4), dtype=np.uint64)
    batch = philox4x32(ctr, (123, 456))
    for i in range(64):
        assert np.array_equal(batch[i], philox4x32(ctr[i], (123, 456)))


def test_pair_draw_layout():
    seed, off = 0x1234_5678_9ABC_DEF0, 0x0000_0002_0000_0003
    K = np.arange(64, dtype=np.int64) + (5 << 35)
    u = pair_draws16(seed, off, K)
    for i, k in enumerate(K):
        q = int(k) >> 3
        words = philox4x32(np.array([q & 0xFFFFFFFF, q >> 32, off & 0xFFFFFFFF, off >> 32], dtype=np.uint64),
                           (seed & 0xFFFFFFFF, seed >> 32))
        w = int(words[(int(k) >> 1) & 3])
        want = (w >> 16) if (int(k) & 1) else (w & 0xFFFF)
        assert int(u[i]) == want


def test_bitrev16():
    assert int(bitrev16(np.array([1]))[0]) == 0x8000
    assert int(bitrev16(np.array([0x00F1]))[0]) == 0x8F00
    x = np.arange(1 << 16, dtype=np.uint32)
    assert np.array_equal(bitrev16(bitrev16(x)), x)
    assert np.array_equal(np.sort(bitrev16(x)), x)     # a permutation of the 16-bit values


def test_draws_are_uniform():
    n = 1 << 20
    bits = pair_draws16(7, 11, np.arange(n, dtype=np.int64)).astype(np.float64)
    mean, sd = bits.mean(), np.sqrt((65536 ** 2 - 1) / 12 / n)
    assert abs(mean - 32767.5) < 5 * sd
    for b in range(16):
        frac = ((bits.astype(np.int64) >> b) & 1).mean()
        assert abs(frac - 0.5) < 5 * 0.5 / np.sqrt(n)
    # different offsets give different streams
    other = pair_draws16(7, 12, np.arange(4096, dtype=np.int64))
    assert np.count_nonzero(other == bits[:4096].astype(np.uint32)) < 4096 * 0.01
    # the reversed draw of a pair's second element is uniform too
    rev = bitrev16(bits.astype(np.uint32)).astype(np.float64)
    assert abs(rev.mean() - 32767.5) < 5 * sd
