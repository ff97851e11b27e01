"""Pins of the oracle's number formats and rounding rules.

Each check compares the oracle with something other than itself: the bit-field
readings printed on the pages, closed-form rounding written a different way
(scale to an integer grid and use numpy's round-half-even), PyTorch's own
float8_e4m3fn conversion, and exhaustive enumeration of the random integer in
stochastic rounding.
"""
import numpy as np
import pytest
import torch

from oracle import formats as F


# --- bit fields printed on the pages ---------------------------------------
def test_widget_bit_fields():
    # Chinese translation, NVFP4 widget: E4M3 0|1101|100 = 96, E2M1 0|11|1 = 6
    assert F.e4m3_decode(0b0_1101_100) == 96.0
    assert F.e2m1_decode(0b0_11_1) == 6.0


def test_e2m1_grid_is_the_pages_set():
    # "Low-precision formats on Blackwell": FP4 holds +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}
    assert sorted(F.E2M1_MAGS.tolist()) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    vals = sorted(F.e2m1_decode(c) for c in range(16))
    assert vals == sorted([-6, -4, -3, -2, -1.5, -1, -0.5, -0.0, 0, 0.5, 1, 1.5, 2, 3, 4, 6])


def test_e4m3_grid_closed_form():
    mags = F.E4M3_MAGS
    assert mags[0] == 0 and mags[1] == 2.0 ** -9 and mags[-1] == 448.0
    assert len(mags) == 127 and np.all(np.diff(mags) > 0)
    # every finite positive E4M3 value is m * 2^k with a 4-bit significand
    expect = set([m * 2.0 ** -9 for m in range(0, 8)])
    for e in range(1, 16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            expect.add((8 + m) * 2.0 ** (e - 10))
    assert set(mags.tolist()) == expect
    assert np.isnan(F.e4m3_decode(0x7F)) and np.isnan(F.e4m3_decode(0xFF))


def test_e4m3_matches_torch_float8_decoding():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    ours = F.decode_e4m3_array(np.arange(256))
    both_nan = np.isnan(ref) & np.isnan(ours)
    assert np.all(both_nan | (ref == ours))


def test_e8m0_values():
    assert F.e8m0_decode(127) == 1.0
    assert F.e8m0_decode(0) == 2.0 ** -127
    assert F.e8m0_decode(254) == 2.0 ** 127


# --- round to nearest ------------------------------------------------------
def _rn_closed_form(v, sub_step, min_normal, max_val, mant_bits):
    """Scale each value to the integer grid of its binade and let numpy's
    round-half-even pick; saturate at max."""
    v = np.asarray(v, dtype=np.float64)
    m = np.abs(v)
    k = np.floor(np.log2(np.maximum(m, min_normal)))
    step = np.where(m < min_normal, sub_step, 2.0 ** (k - mant_bits))
    q = np.round(m / step) * step
    q = np.minimum(q, max_val)
    return np.copysign(q, v)


def _probe_values(mags):
    mids = (mags[1:] + mags[:-1]) / 2
    pts = np.concatenate([mags, mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
                          np.nextafter(mids.astype(np.float32), np.float32(-np.inf)),
                          mags[-1] * np.array([1.01, 1.5, 3.0, 1e6])])
    rng = np.random.default_rng(0)
    pts = np.concatenate([pts, rng.uniform(0, mags[-1] * 1.2, 20000)]).astype(np.float32)
    return np.concatenate([pts, -pts])


def test_rn_e2m1_against_closed_form():
    v = _probe_values(F.E2M1_MAGS)
    ours = F.decode_e2m1_array(F.rn_code(v, F.E2M1_TABLE))
    ref = _rn_closed_form(v, 0.5, 1.0, 6.0, 1)
    assert np.array_equal(ours, ref)


def test_rn_e2m1_ties_and_the_3p2_example():
    # "3.2 ... nearest values our format can represent are 3 and 4. Rounding to
    # 3 introduces a quantization error of -0.2"
    c = F.rn_code(np.float32(3.2), F.E2M1_TABLE)
    assert F.e2m1_decode(int(c)) == 3.0
    assert abs(3.0 - float(np.float32(3.2)) - (-0.2)) < 1e-6
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for x, want in ties.items():
        assert F.e2m1_decode(int(F.rn_code(np.float32(x), F.E2M1_TABLE))) == want
    # signed zero is kept
    assert int(F.rn_code(np.float32(-0.1), F.E2M1_TABLE)) == 0x8


def test_rn_e4m3_against_closed_form():
    v = _probe_values(F.E4M3_MAGS)
    ours = F.decode_e4m3_array(F.rn_code(v, F.E4M3_TABLE))
    ref = _rn_closed_form(v, 2.0 ** -9, 2.0 ** -6, 448.0, 3)
    assert np.array_equal(ours, ref)


def test_rn_e4m3_against_torch_float8_cast():
    v = _probe_values(F.E4M3_MAGS)
    v = v[np.abs(v) <= 448.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = F.rn_code(v, F.E4M3_TABLE)
    assert np.array_equal(ours, ref)


# --- stochastic rounding -----------------------------------------------------
def test_sr_page_example_exhaustive():
    # "Re-quantization with stochastic rounding": 4.5 re-quantized with scale 2
    # is 2.25 on the FP4 grid and becomes 2 three quarters of the time, 3 a
    # quarter of the time -- over all 2^16 random integers exactly.
    r = np.arange(1 << 16)
    w = np.full(r.shape, np.float32(4.5 / 2))
    vals = F.decode_e2m1_array(F.sr_code(w, F.E2M1_TABLE, r))
    assert np.count_nonzero(vals == 2.0) == 49152
    assert np.count_nonzero(vals == 3.0) == 16384
    assert 2 * vals.mean() == 4.5


@pytest.mark.parametrize("table", [F.E2M1_TABLE, F.E4M3_TABLE], ids=["e2m1", "e4m3"])
def test_sr_expectation_exhaustive(table):
    """Over all 2^16 random integers the mean is a + (b-a) floor(f 2^16)/2^16:
    exact when f is a multiple of 2^-16, below |w| by < 2^-16 (b-a) otherwise;
    the result is always one of the two neighbours."""
    mags, _, _ = table
    decode = F.decode_e2m1_array if mags[-1] == 6 else F.decode_e4m3_array
    rng = np.random.default_rng(1)
    ws = rng.uniform(0, mags[-1], 12).astype(np.float32)
    ws = np.concatenate([ws, [np.float32(mags[3] + (mags[4] - mags[3]) * 0.375)]])
    r = np.arange(1 << 16)
    for w in ws:
        vals = decode(F.sr_code(np.full(r.shape, w, dtype=np.float32), table, r))
        a = mags[mags <= w].max()
        b = mags[mags > w].min()
        assert set(np.unique(vals)) <= {a, b}
        bias = vals.mean() - float(w)
        assert -(b - a) * 2.0 ** -16 < bias <= 0.0
        f = (float(w) - a) / (b - a)
        if (f * 65536) == int(f * 65536):
            assert bias == 0.0
    # negative values mirror, saturation takes no randomness
    neg = decode(F.sr_code(np.full(r.shape, -ws[0], dtype=np.float32), table, r))
    pos = decode(F.sr_code(np.full(r.shape, ws[0], dtype=np.float32), table, r))
    assert np.array_equal(neg, -pos)
    sat = decode(F.sr_code(np.full(16, mags[-1] * 1.05, dtype=np.float32), table, np.arange(16)))
    assert np.all(sat == mags[-1])


def test_bf16_helpers_roundtrip():
    x = torch.randn(1000, generator=torch.Generator().manual_seed(0)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    f = F.bf16_to_f32(bits)
    assert np.array_equal(f, x.float().numpy())
    y = torch.randn(1000, generator=torch.Generator().manual_seed(1))
    assert np.array_equal(F.f32_to_bf16_rne(y.numpy()), y.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
