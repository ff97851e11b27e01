"""Pins of the Four Over Six reading ("Recipe details": the activation
quantizer selects between two scale factors per block; the selection rule is
not on the pages, so this function is parity unpinned as to the rule itself).
What is pinned is that the oracle does what the reading says: the kept
candidate's exact (float64) error never exceeds the plain quantizer's, blocks
that the 4-mapping represents exactly take 4 with zero error, blocks that the
6-mapping represents exactly keep 6, zero blocks keep 6, the total error on
Gaussian data is below the plain quantizer's, and a planted "keep the larger
error" rule fails the first pin."""
import numpy as np

from oracle import nvfp4 as NV


def _err64(x, codes, scales, sg):
    d = NV.dequantize_f64(codes, scales, sg)
    return ((np.asarray(x, np.float64) - d) ** 2).reshape(x.shape[0], -1, 16).sum(-1)


def test_kept_candidate_never_worse_than_plain():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((128, 256)) * np.exp(rng.uniform(-3, 3, (128, 1)))).astype(np.float32)
    c, s, sg = NV.quantize_four_over_six(x)
    cp, sp, sgp = NV.quantize(x)
    assert sg == sgp
    e46, e6 = _err64(x, c, s, sg), _err64(x, cp, sp, sg)
    # the decision is taken on fp32 sums: allow their rounding, nothing more
    assert np.all(e46 <= e6 * (1 + 1e-5) + 1e-30)
    assert np.sum(e46 < e6) > 0.2 * e6.size          # many blocks gain


def test_exact_blocks_choose_their_mapping():
    # with sg = 1 a block whose maximum is 4 and whose values sit on the E2M1
    # grid is exact under the 4-mapping (scale 1) but not under 6 (scale
    # RN_E4M3(4/6) = 0.6875): it takes 4, error 0
    b4 = np.array([4, 3, 2, 1.5, 1, 0.5, 0, -4, -3, -2, -1.5, -1, -0.5, 0, 3, 2], np.float32)
    # a block exact under the 6-mapping (scale 1) keeps 6
    b6 = np.array([6, 4, 3, 2, 1.5, 1, 0.5, 0, -6, -4, -3, -2, -1.5, -1, -0.5, 0], np.float32)
    z = np.zeros(16, np.float32)
    x = np.stack([b4, b6, z])
    c, s, _, take4 = NV.quantize_four_over_six(x, sg=1.0, return_choice=True)
    assert list(take4[:, 0]) == [True, False, False]
    assert np.all(_err64(x, c, s, np.float32(1.0)) == 0)
    assert s[2, 0] == 0


def test_total_error_below_plain_nvfp4():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((256, 512)).astype(np.float32)
    c, s, sg = NV.quantize_four_over_six(x)
    cp, sp, _ = NV.quantize(x)
    assert _err64(x, c, s, sg).sum() < 0.97 * _err64(x, cp, sp, sg).sum()


def test_planted_larger_error_rule_fails():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((32, 128)).astype(np.float32)
    sg = NV.outer_scale(x)
    xb = x.reshape(-1, 16)
    c6, s6 = NV._quantize_blocks(xb, sg, 6.0)
    c4, s4 = NV._quantize_blocks(xb, sg, 4.0)
    wrong4 = NV.block_sq_error_f32(xb, c4, s4, sg) > NV.block_sq_error_f32(xb, c6, s6, sg)
    cw = np.where(wrong4[:, None], c4, c6).reshape(x.shape)
    sw = np.where(wrong4, s4, s6).reshape(32, 8)
    cp, sp, _ = NV.quantize(x)
    assert not np.all(_err64(x, cw, sw, sg) <= _err64(x, cp, sp, sg) * (1 + 1e-5) + 1e-30)


def test_error_sum_order_is_sequential_fp32():
    # sixteen squares whose sum depends on the order in fp32: the function
    # must add them in index order
    xb = np.zeros((1, 16), np.float32)
    xb[0, 0] = 1.0
    xb[0, 1:] = 2.0 ** -12
    codes = np.zeros((1, 16), np.uint8)
    s_code = np.array([0], np.uint8)                  # scale 0: d = 0, e = x
    got = NV.block_sq_error_f32(xb, codes, s_code, np.float32(1.0))[0]
    acc = np.float32(0.0)
    for v in xb[0]:
        acc = np.float32(acc + np.float32(v * v))
    assert got == acc and got == np.float32(1.0)      # each 2^-24 is lost against 1.0 in order
