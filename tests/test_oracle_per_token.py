"""Pins of the per-token (per-row) outer scale ("Recipe details": one FP32
scale per token for activations, chosen for batch invariance).  The oracle's
per-row quantizer is checked against the per-tensor quantizer applied to each
row as its own tensor, against batch invariance (another row's values never
change a row's codes, which the per-tensor scale does not satisfy), against
the per-tensor result when every row has the same largest magnitude, and
against the scale rule's fixed point (each non-zero row's largest block gets
the E4M3 maximum 448)."""
import numpy as np
import pytest

from oracle import layout as L
from oracle import nvfp4 as NV
from oracle import requant as RQ

E4M3_448 = 0x7E


def _x(rows=12, cols=96, seed=0):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-6, 6, (rows, 1)))).astype(np.float32)
    x[3] = 0.0                       # an all-zero token
    x[5, 17] = 5000.0                # an outlier token
    x[7, :16] = 0.0                  # a zero block inside a non-zero token
    return x


def test_each_row_equals_the_per_tensor_quantizer_on_that_row():
    x = _x()
    c, s, sg = NV.quantize_rows(x)
    for r in range(x.shape[0]):
        cr, sr, sgr = NV.quantize(x[r:r + 1])
        assert sg[r] == sgr
        assert np.array_equal(c[r:r + 1], cr) and np.array_equal(s[r:r + 1], sr)


def test_batch_invariance_and_per_tensor_contrast():
    x = _x(seed=1)
    y = x.copy()
    y[2] *= 1000.0                   # another token changes, and becomes the tensor's largest
    y[2, 0] = 100.0 * np.abs(x).max()
    c0, s0, _ = NV.quantize_rows(x)
    c1, s1, _ = NV.quantize_rows(y)
    keep = np.arange(x.shape[0]) != 2
    assert np.array_equal(c0[keep], c1[keep]) and np.array_equal(s0[keep], s1[keep])
    # the per-tensor scale is not batch invariant: the same change moves other rows
    t0 = NV.quantize(x)
    t1 = NV.quantize(y)
    assert not np.array_equal(t0[1][keep], t1[1][keep])


def test_equal_row_amax_gives_the_per_tensor_result():
    rng = np.random.default_rng(2)
    x = rng.uniform(-1, 1, (6, 64)).astype(np.float32)
    x[:, 5] = 3.0                    # every row's largest magnitude is 3
    c, s, sg = NV.quantize_rows(x)
    ct, st, sgt = NV.quantize(x)
    assert np.all(sg == sgt) and np.array_equal(c, ct) and np.array_equal(s, st)


def test_scale_fixed_point_zero_rows_and_error_bound():
    x = _x(seed=3)
    c, s, sg = NV.quantize_rows(x)
    nz = np.any(x != 0, axis=1)
    # amax_r / fp32(6 sg_r) rounds to 448: each non-zero row holds the E4M3 maximum
    assert np.all(np.any(s[nz] == E4M3_448, axis=1))
    assert np.all(sg[~nz] == 1.0) and np.all(s[~nz] == 0) and np.all((c[~nz] & 7) == 0)
    # |x - deq| <= one block-scale unit (the largest E2M1 gap is 2, so half of it)
    deq = NV.dequantize_rows_f64(c, s, sg)
    unit = NV.dequantize_rows_f64(np.full_like(c, 2), s, sg)        # E2M1 code 2 = 1.0
    assert np.all(np.abs(deq - x) <= unit + 1e-30)
    # the f32 dequantization is the f64 one rounded once
    assert np.array_equal(NV.dequantize_rows_f32(c, s, sg), deq.astype(np.float32))


def test_planted_column_scale_fails_the_row_pin():
    x = _x(seed=4)
    c, s, sg = NV.quantize_rows(x)
    wrong = np.repeat(NV.outer_scale_rows(x.T)[: x.shape[0]], 1)   # scales from the columns
    cw, sw, _ = NV.quantize_rows(x, wrong)
    assert not (np.array_equal(cw, c) and np.array_equal(sw, s))


def test_requant_rows_reduces_to_per_tensor_with_a_shared_scale():
    rng = np.random.default_rng(5)
    go = np.array([0, 37, 37, 130], dtype=np.int64)
    x = rng.standard_normal((130, 128)).astype(np.float32)
    c, s, sg = NV.quantize(x)
    P = L.padded_cap(130, 3)
    a = RQ.requant_grouped(c, s, sg, go, seed=9, offset=2, P_cols=P)
    b = RQ.requant_grouped_rows(c, s, np.full(130, sg, np.float32), go, seed=9, offset=2, P_cols=P)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # per-row scales enter the transposed blocks value by value
    cr, sr, sgr = NV.quantize_rows(x)
    d = RQ.requant_grouped_rows(cr, sr, sgr, go, seed=9, offset=2, P_cols=P)
    e = RQ.transposed_grouped_sr(NV.dequantize_rows_f32(cr, sr, sgr), go, 9, 2, P)
    assert np.array_equal(d[0], e[0]) and np.array_equal(d[1], e[1])


@pytest.mark.parametrize("r", [0, 5, 11])
def test_dequantize_rows_matches_per_row_dequantize(r):
    x = _x(seed=6)
    c, s, sg = NV.quantize_rows(x)
    assert np.array_equal(NV.dequantize_rows_f64(c, s, sg)[r], NV.dequantize_f64(c[r], s[r], sg[r]))
