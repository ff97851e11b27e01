"""Pins of the RHT-32 + block-scaled S2F6 oracle ("Quantized communications"):
the Hadamard matrix against the Walsh closed form, orthogonality and energy
preservation (the pages: total energy unchanged, exact inverse), the fp32
butterfly against the closed form within its rounding bound, the S2F6 grid
the pages state (k/64, -128/64 .. 127/64), nearest-value rounding against a
brute-force search of that grid, the scale rule's special cases, and the
8.25 bits per value."""
import numpy as np
import pytest

from oracle import rht as R


def _walsh(n=32):
    i = np.arange(n)
    bits = np.bitwise_and.outer(i, i)
    pop = np.array([[bin(int(b)).count("1") for b in row] for row in bits])
    return np.where(pop % 2 == 0, 1, -1)


def test_hadamard_is_the_walsh_matrix_and_orthogonal():
    H = R.hadamard()
    assert H.shape == (32, 32)
    assert np.array_equal(H, _walsh())
    assert np.array_equal(H @ H.T, 32 * np.eye(32, dtype=np.int64))


@pytest.mark.parametrize("mask", [0, 0xFFFFFFFF, 0x12345678, 0x80000001])
def test_rht_f64_matches_closed_form_preserves_energy_and_inverts(mask):
    rng = np.random.default_rng(mask & 0xFFFF)
    x = rng.standard_normal((5, 96)) * 100.0
    d = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(32)])
    W = _walsh()
    want = np.stack([np.concatenate([W @ (d * blk) / np.sqrt(32) for blk in row.reshape(-1, 32)]) for row in x])
    y = R.rht_f64(x, mask)
    assert np.allclose(y, want, rtol=0, atol=1e-9)
    # energy of every block unchanged; the inverse recovers the input
    assert np.allclose((y.reshape(5, 3, 32) ** 2).sum(-1), (x.reshape(5, 3, 32) ** 2).sum(-1), rtol=1e-12)
    assert np.allclose(R.irht_f64(y, mask), x, rtol=0, atol=1e-9)


def test_energy_example_shape():
    """The pages' illustration: 32 values on [-500, 500], 4 of them outliers;
    an orthonormal Hadamard transform keeps the energy and lowers the peak."""
    rng = np.random.default_rng(3)
    x = rng.uniform(-60, 60, 32)
    x[[3, 11, 20, 29]] = [310.0, -280.0, 250.0, -300.0]
    y = R.rht_f64(x, 0)
    assert np.isclose((y ** 2).sum(), (x ** 2).sum(), rtol=1e-12)
    assert np.abs(y).max() < np.abs(x).max()


def test_fp32_butterfly_within_rounding_bound_of_the_definition():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((64, 128)) * np.exp(rng.uniform(-8, 8, (64, 128)))).astype(np.float32)
    for mask in (0, 0xA5A5A5A5):
        y32 = R.rht_f32(x, mask).astype(np.float64)
        y64 = R.rht_f64(x.astype(np.float64), mask)
        # five rounded additions and one rounded multiply per output
        bound = 7 * 2.0 ** -24 * np.abs(x.reshape(64, 4, 32)).sum(-1, keepdims=True) / np.sqrt(32)
        assert np.all(np.abs(y32 - y64).reshape(64, 4, 32) <= bound + 1e-30)
        back = R.irht_f32(R.rht_f32(x, mask), mask).astype(np.float64)
        assert np.all(np.abs(back - x).reshape(64, 4, 32) <= 2 * bound + 1e-30)


def test_planted_butterfly_sign_error_is_caught():
    """A (a - b, a + b) butterfly (swapped outputs) must fail the closed form."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 32)).astype(np.float32)
    v = x.copy()
    h = 1
    while h < 32:
        idx = np.arange(32)
        lo = idx[(idx & h) == 0]
        a, b = v[:, lo].copy(), v[:, lo + h].copy()
        v[:, lo], v[:, lo + h] = a - b, a + b
        h *= 2
    assert not np.allclose(v * R.INV_SQRT32_F32, R.rht_f64(x.astype(np.float64), 0), atol=1e-4)


def test_s2f6_grid_is_the_pages_range():
    v = R.s2f6_values()
    assert v.size == 256 and v[0] == -2.0 and v[-1] == 127 / 64
    assert np.allclose(np.diff(v), 1 / 64)


def test_s2f6_rounding_is_nearest_with_ties_to_even_against_brute_force():
    rng = np.random.default_rng(4)
    blocks = rng.standard_normal((200, 32)).astype(np.float32) * np.float32(3.7)
    codes, scales = R.s2f6_quantize(blocks)
    e = scales.astype(np.int64) - 127          # [200, 1]: one block per row
    grid = R.s2f6_values()
    w = blocks.astype(np.float64) * np.ldexp(1.0, -e)
    # nearest grid value; ties (exact halves) to the even code
    dist = np.abs(w[..., None] - grid)
    best = dist.min(-1, keepdims=True)
    cand = np.where(dist == best, np.arange(-128, 128), 10 ** 6)
    even = np.where(cand % 2 == 0, cand, 10 ** 6).min(-1)
    want = np.where((dist == best).sum(-1) > 1, even, cand.min(-1))
    assert np.array_equal(codes.astype(np.int64), want)
    # the block maximum maps into [1, 2): its code is in [64, 128) before saturation
    am = np.abs(w).max(-1)
    assert np.all((am >= 1) & (am < 2))


def test_s2f6_ties_saturation_zero_block_and_size():
    e0 = np.zeros((1, 32), np.float32)
    c, s = R.s2f6_quantize(e0)
    assert s[0, 0] == 0 and np.all(c == 0)
    # block max 1.5 -> scale 2^0; 0.5/64 ties to 0, 1.5/64 ties to 2, 1.99 saturates to 127
    b = np.zeros((1, 32), np.float32)
    b[0, :4] = [1.5, 0.5 / 64, 1.5 / 64, -2.5 / 64]
    c, s = R.s2f6_quantize(b)
    assert s[0, 0] == 127 and list(c[0, :4]) == [96, 0, 2, -2]
    b[0, 0] = 1.99
    c, s = R.s2f6_quantize(b)
    assert c[0, 0] == 127
    # 8-bit codes plus one 8-bit scale per 32 values: 8.25 bits per value
    x = np.ones((3, 64), np.float32)
    c, s = R.s2f6_quantize(x)
    assert (c.nbytes + s.nbytes) * 8 / x.size == 8.25


def test_round_trip_error_is_half_a_step():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((32, 256)) * 10).astype(np.float32)
    c, s = R.s2f6_quantize(x)
    back = R.s2f6_dequantize(c, s).astype(np.float64)
    step = np.ldexp(1.0, s.astype(np.int64) - 127 - 6)[..., None]
    err = np.abs(back - x).reshape(32, 8, 32)
    # elements past the largest code (|v| / 2^e above 127.5 / 64) saturate
    sat = np.abs(x).reshape(32, 8, 32) / (step * 64) > 127.5 / 64
    assert np.all(err[~sat] <= (step / 2 + np.zeros_like(err))[~sat] + 1e-30)
    assert np.all(c.reshape(32, 8, 32)[sat] != 0)
