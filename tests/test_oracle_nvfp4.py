"""Pins of the oracle's NVFP4 quantizer against the pages' worked examples,
closed forms and figure counts (End-to-End 4-Bit Training)."""
import json
import os

import numpy as np
import pytest

from oracle import formats as F
from oracle import nvfp4 as NV
from precision_moe_numerics_nvfp4_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _block(vals):
    b = np.zeros((1, 16), dtype=np.float32)
    b[0, :len(vals)] = vals
    return b


def test_worked_example_593p7():
    g = _load("nvfp4_examples.json")["593.7"]
    codes, scales, _ = NV.quantize(_block([np.float32(g["input"])]), sg=1.0)
    assert int(scales[0, 0]) == int(g["scale_code"], 16)
    assert F.e4m3_decode(int(scales[0, 0])) == g["scale"]
    assert int(codes[0, 0]) == int(g["code"], 16)
    deq = NV.dequantize_f64(codes, scales, 1.0)[0, 0]
    assert deq == g["value"]
    assert abs((deq - np.float32(g["input"])) - g["error"]) < 0.05


def test_worked_example_minus54_and_5p4():
    g = _load("nvfp4_examples.json")
    blk = _block([np.float32(-54.0), np.float32(5.4), np.float32(1.0)])
    codes, scales, _ = NV.quantize(blk, sg=1.0)
    e = g["-54"]
    assert F.e4m3_decode(int(scales[0, 0])) == e["scale"] and int(scales[0, 0]) == int(e["scale_code"], 16)
    assert F.e2m1_decode(int(codes[0, 0])) == e["fp4"]
    f = g["5.4"]
    assert F.e2m1_decode(int(codes[0, 1])) == f["fp4"]
    assert NV.dequantize_f64(codes, scales, 1.0)[0, 1] == f["value"]
    # the bf16 neighbour of 5.4 lands on the same code
    blk[0, 1] = np.float32(5.40625)
    codes2, _, _ = NV.quantize(blk, sg=1.0)
    assert codes2[0, 1] == codes[0, 1]


def test_representable_range_and_outer_scale_shift():
    g = _load("nvfp4_examples.json")["range"]
    e2 = F.E2M1_MAGS[F.E2M1_MAGS > 0]
    e4 = F.E4M3_MAGS[F.E4M3_MAGS > 0]
    prods = (e2[:, None] * e4[None, :]).reshape(-1)
    assert prods.min() == 2.0 ** g["min_log2"] and prods.max() == g["max"]
    prods2 = prods * 2.0
    assert prods2.min() == 2.0 ** g["min_log2_sg2"] and prods2.max() == g["max_sg2"]


def test_outer_scale_maps_amax_to_6_times_448():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((8, 64)) * 0.02).astype(np.float32)
    sg = NV.outer_scale(x)
    assert sg == np.float32(np.abs(x).max() / np.float32(2688))
    codes, scales, _ = NV.quantize(x, sg)
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert F.e4m3_decode(int(scales[i[0], i[1] // 16])) == 448.0
    assert abs(F.e2m1_decode(int(codes[i]))) == 6.0
    assert NV.outer_scale(np.zeros((2, 16), np.float32)) == 1.0


def test_all_zero_block_and_signed_zero():
    blk = np.zeros((1, 32), dtype=np.float32)
    blk[0, 3] = -0.0
    blk[0, 16:] = np.linspace(-1, 1, 16)
    codes, scales, _ = NV.quantize(blk, sg=1.0)
    assert scales[0, 0] == 0 and np.all(codes[0, :16] & 7 == 0)
    assert codes[0, 3] == 0x8 and codes[0, 0] == 0x0


def test_block_error_bound_and_saturation_free():
    """With the RN scale the block maximum maps to within one E4M3 step of
    6, and every element is within half an E2M1 gap (at most 1) of the grid."""
    rng = np.random.default_rng(5)
    x = (rng.standard_t(3, size=(64, 256)) * 0.05).astype(np.float32)
    sg = NV.outer_scale(x)
    codes, scales, _ = NV.quantize(x, sg)
    deq = NV.dequantize_f64(codes, scales, sg)
    step = F.decode_e4m3_array(np.repeat(scales, 16, axis=1)) * float(sg)
    assert np.all(np.abs(deq - x) <= step * 1.0 + 1e-30 + np.maximum(0, np.abs(x) - 6 * step))


def test_dequant_f32_is_one_rounding_of_exact():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((16, 64)).astype(np.float32)
    codes, scales, sg = NV.quantize(x)
    assert np.array_equal(NV.dequantize_f32(codes, scales, sg),
                          NV.dequantize_f64(codes, scales, sg).astype(np.float32))


def test_pack_layout():
    codes = np.arange(32, dtype=np.uint8).reshape(2, 16) & 0xF
    p = NV.pack(codes)
    assert p[0, 0] == 0x10 and p[0, 1] == 0x32 and p[1, 7] == 0xFE
    assert np.array_equal(NV.unpack(p), codes)


def test_figure2_full_large_row():
    # "Block-scaled backward passes", Figure 2: 1x16 row scales keep all 256
    # values; 16x1 column scales keep the large row and 19 small values and
    # round the other 221 to zero.
    g = _load("figure_counts.json")["figure2"]
    t = W.fig2_tile()
    c_row, s_row, _ = NV.quantize(t, sg=1.0)
    c_col, s_col, _ = NV.quantize_col16(t, sg=1.0)
    kept_row = np.count_nonzero(NV.dequantize_f64(c_row, s_row, 1.0))
    deq_col = NV.dequantize_f64(c_col.T, s_col.T, 1.0).T
    kept_col = np.count_nonzero(deq_col)
    assert kept_row == g["kept_1x16"]
    assert kept_col == g["kept_16x1"]
    assert np.count_nonzero(deq_col[0]) == 16
    assert np.count_nonzero(deq_col[1:]) == g["small_kept_16x1"]
    assert 256 - kept_col == g["zeroed_16x1"]


def test_figure3_single_outlier():
    # Figure 3: 1x16 keeps 241 of 256 (the outlier's group flushes to zero
    # around it); one 16x16 scale keeps only the outlier.
    g = _load("figure_counts.json")["figure3"]
    t = W.fig3_tile()
    c_row, s_row, _ = NV.quantize(t, sg=1.0)
    c_t, s_t, _ = NV.quantize_tile16x16(t, sg=1.0)
    assert np.count_nonzero(NV.dequantize_f64(c_row, s_row, 1.0)) == g["kept_1x16"]
    deq_t = NV.dequantize_tile16x16_f64(c_t, s_t, 1.0)
    assert np.count_nonzero(deq_t) == g["kept_16x16"]
    assert deq_t[t == 64.0].item() != 0


@pytest.mark.parametrize("mistake", ["dropped_six", "ties_to_odd", "transposed_blocks"])
def test_pins_catch_planted_mistakes(monkeypatch, mistake):
    """A plausible slip planted in the oracle must break one of the pins."""
    from tests import test_oracle_formats as TF
    if mistake == "dropped_six":
        orig = NV._quantize_blocks
        monkeypatch.setattr(NV, "_quantize_blocks", lambda xb, sg: orig(xb, np.float32(sg) / np.float32(6.0)))
        pin = test_worked_example_593p7
    elif mistake == "ties_to_odd":
        orig_rn = F.rn_code

        def bad_rn(v, table):
            c = orig_rn(v, table)
            x = np.abs(np.asarray(v, dtype=np.float64))
            return np.where(x == 0.75, np.uint8(1), c)
        monkeypatch.setattr(F, "rn_code", bad_rn)
        pin = TF.test_rn_e2m1_ties_and_the_3p2_example
    else:
        orig_q = NV.quantize
        monkeypatch.setattr(NV, "quantize", lambda x, sg=None: tuple(
            (r.T if i < 2 and r.ndim == 2 and r.shape[0] == r.shape[1] else r)
            for i, r in enumerate(orig_q(np.asarray(x).T, sg))))
        pin = test_figure2_full_large_row
    with pytest.raises(AssertionError):
        pin()
