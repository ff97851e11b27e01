"""RHT-32 + block-scaled S2F6 on the GPU against the oracle: codes and scales
bit-exact (the oracle takes the transform in the kernel's fp32 order), the
inverse bit-exact in fp32 and bf16, ragged row counts, zero blocks, outlier
blocks and several sign masks; the round trip stays within the quantization
step plus the transform's rounding."""
import numpy as np
import pytest
import torch

from oracle import rht as R
from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
from tests.gpu_helpers import bf16_f32, check_status, dev, gempty, gfull

pytestmark = pytest.mark.gpu


def _x(rows, cols, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn((rows, cols), generator=g, device="cuda") * 3.0
    if rows > 2:
        x[1, :32] = 0.0                      # a zero block
        x[2, 5] = 4000.0                     # an outlier block
        x[0, 32:64] = 1e-30                  # a tiny block (subnormal range after scaling)
    if rows > 5 and cols >= 160:
        # the far ends of the scale range: a huge block (scale near 127, the
        # inverse's large-exponent path), a block of fp32 subnormals (scale
        # clamped at -127), and a block whose small values turn subnormal
        # after the 1/sqrt(32) multiply while the block max stays normal
        x[3, 64:96] = torch.randn(32, generator=g, device="cuda") * 1e36
        x[4, 96:128] = torch.randn(32, generator=g, device="cuda") * 1e-39
        x[5, 128:160] = torch.randn(32, generator=g, device="cuda") * 1e-40
        x[5, 128:132] = 3e-34
    return x.to(torch.bfloat16).contiguous()


@pytest.mark.parametrize("rows,cols,mask", [(1, 32, 0), (3, 64, 0xFFFFFFFF), (37, 256, 0x9E3779B9),
                                            (129, 4096, 0x12345678), (5, 96, 0x80000001)])
def test_quantize_and_inverse_match_oracle(rows, cols, mask):
    x = _x(rows, cols, seed=rows + cols)
    codes = gfull((rows, cols), 0x55, dtype=torch.int8, device=dev())
    scales = gfull((rows, cols // 32), 0xAA, dtype=torch.uint8, device=dev())
    N.rht32_s2f6_quantize(x, rows, cols, mask, codes, scales)
    y32 = gempty((rows, cols), dtype=torch.float32, device=dev())
    y16 = gempty((rows, cols), dtype=torch.bfloat16, device=dev())
    N.s2f6_dequantize_rht32_inverse(codes, scales, rows, cols, mask, y32, N.NV_OUT_FP32)
    N.s2f6_dequantize_rht32_inverse(codes, scales, rows, cols, mask, y16, N.NV_OUT_BF16)
    check_status()
    xf = bf16_f32(x)
    want_c, want_s = R.rht_s2f6_quantize(xf, mask)
    assert np.array_equal(codes.cpu().numpy(), want_c)
    assert np.array_equal(scales.cpu().numpy(), want_s)
    back = R.s2f6_dequantize_irht(want_c, want_s, mask)
    assert np.array_equal(y32.cpu().numpy().view(np.uint32), back.view(np.uint32))
    want16 = torch.from_numpy(back).to(torch.bfloat16)
    assert torch.equal(y16.cpu().view(torch.int16), want16.view(torch.int16))
    # round trip: within half a quantization step (in the rotated basis; the
    # orthonormal inverse keeps the Euclidean error) plus transform rounding
    err = np.abs(back.astype(np.float64) - xf).reshape(rows, -1, 32)
    step = np.ldexp(1.0, want_s.astype(np.int64) - 127 - 6)[..., None]
    yq = R.rht_f32(xf, mask).reshape(rows, -1, 32).astype(np.float64)
    unsat = np.all(np.abs(yq) / (step * 64) <= 127.5 / 64, axis=-1)
    e2 = np.sqrt((err ** 2).sum(-1))
    bound = np.sqrt(32) * step[..., 0] / 2 + 1e-5 * np.sqrt((xf.astype(np.float64).reshape(rows, -1, 32) ** 2).sum(-1)) + 1e-30
    assert np.all(e2[unsat] <= bound[unsat])


def test_rejects_bad_arguments():
    x = torch.zeros((2, 48), dtype=torch.bfloat16, device=dev())
    c = torch.zeros((2, 48), dtype=torch.int8, device=dev())
    s = torch.zeros((2, 2), dtype=torch.uint8, device=dev())
    with pytest.raises(N.NvError):
        N.rht32_s2f6_quantize(x, 2, 48, 0, c, s)          # cols % 32
    with pytest.raises(N.NvError):
        N.s2f6_dequantize_rht32_inverse(c, s, 2, 32, 0, x, 7)  # bad dtype


def test_misaligned_pointers_are_rejected_and_nothing_is_written():
    rows, cols = 4, 64
    xb = torch.zeros(rows * cols + 16, dtype=torch.bfloat16, device=dev())
    cb = gfull((rows * cols + 32,), 0x55, dtype=torch.int8, device=dev())
    s = gfull((rows, cols // 32), 0xAA, dtype=torch.uint8, device=dev())
    yb = gfull((rows * cols + 16,), 7.0, dtype=torch.float32, device=dev())
    with pytest.raises(N.NvError):
        N.rht32_s2f6_quantize(xb[8:8 + rows * cols], rows, cols, 0, cb[:rows * cols], s)   # x 16-byte aligned
    with pytest.raises(N.NvError):
        N.rht32_s2f6_quantize(xb[:rows * cols], rows, cols, 0, cb[16:16 + rows * cols], s)  # codes 16-byte aligned
    with pytest.raises(N.NvError):
        N.s2f6_dequantize_rht32_inverse(cb[:rows * cols], s, rows, cols, 0, yb[4:4 + rows * cols], N.NV_OUT_FP32)
    torch.cuda.synchronize()
    assert torch.all(cb == 0x55) and torch.all(s == 0xAA) and torch.all(yb == 7.0)
    check_status()


def test_empty_inputs_are_no_ops():
    c = gfull((64,), 0x55, dtype=torch.int8, device=dev())
    s = gfull((2,), 0xAA, dtype=torch.uint8, device=dev())
    x = torch.zeros((64,), dtype=torch.bfloat16, device=dev())
    N.rht32_s2f6_quantize(x, 0, 64, 1, c, s)
    N.s2f6_dequantize_rht32_inverse(c, s, 2, 0, 1, x, N.NV_OUT_BF16)
    torch.cuda.synchronize()
    assert torch.all(c == 0x55) and torch.all(s == 0xAA) and torch.all(x == 0)
    check_status()


def test_full_size_sampled_rows_match_oracle():
    """The combine activations at full size ([131072 x 4096] bf16, the launch
    the benchmark times): every code and scale of 48 sampled rows, and their
    inverse, bit-exact against the oracle."""
    rows, cols, mask = 131072, 4096, 0x6A09E667
    g = torch.Generator(device="cuda").manual_seed(11)
    x = (torch.randn((rows, cols), generator=g, device="cuda") * 2.0).to(torch.bfloat16)
    codes = gempty((rows, cols), dtype=torch.int8, device=dev())
    scales = gempty((rows, cols // 32), dtype=torch.uint8, device=dev())
    N.rht32_s2f6_quantize(x, rows, cols, mask, codes, scales)
    y = gempty((rows, cols), dtype=torch.bfloat16, device=dev())
    N.s2f6_dequantize_rht32_inverse(codes, scales, rows, cols, mask, y, N.NV_OUT_BF16)
    check_status()
    pick = torch.cat([torch.tensor([0, rows - 1]), torch.randint(1, rows - 1, (46,), generator=torch.Generator().manual_seed(5))])
    pick_d = pick.to(dev())
    xs = bf16_f32(x[pick_d])
    want_c, want_s = R.rht_s2f6_quantize(xs, mask)
    assert np.array_equal(codes[pick_d].cpu().numpy(), want_c)
    assert np.array_equal(scales[pick_d].cpu().numpy(), want_s)
    back = torch.from_numpy(R.s2f6_dequantize_irht(want_c, want_s, mask)).to(torch.bfloat16)
    assert torch.equal(y[pick_d].cpu().view(torch.int16), back.view(torch.int16))


def _w2_operands(sizes, N_, K, seed):
    from precision_moe_numerics_nvfp4_gb300.pipeline import NvTensor
    o = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    go = torch.from_numpy(o).to(dev())
    M, E = int(o[-1]), len(sizes)
    g = torch.Generator(device="cuda").manual_seed(seed)
    h = torch.randn((M, K), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((E, N_, K), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    hq, wq = NvTensor(1, M, K, dev(), E=E), NvTensor(E, N_, K, dev())
    hq.quantize(h, go)
    wq.quantize(w)
    return go, M, E, hq, wq


def _fused_vs_separate(sizes, N_, K, mask, with_y):
    go, M, E, hq, wq = _w2_operands(sizes, N_, K, seed=M_seed(sizes))
    y_ref = gempty((M, N_), dtype=torch.bfloat16, device=dev())
    N.grouped_gemm_nvfp4_fwd(None, hq.sg, hq.codes, hq.scales, wq.codes, wq.scales, wq.sg, go, E, M, N_, K, y_ref,
                             N.NV_OUT_BF16)
    c_ref = gempty((M, N_), dtype=torch.int8, device=dev())
    s_ref = gempty((M, N_ // 32), dtype=torch.uint8, device=dev())
    N.rht32_s2f6_quantize(y_ref, M, N_, mask, c_ref, s_ref)
    y = gfull((M, N_), 7.0, dtype=torch.bfloat16, device=dev()) if with_y else None
    c = gfull((M, N_), 0x55, dtype=torch.int8, device=dev())
    s = gfull((M, N_ // 32), 0xAA, dtype=torch.uint8, device=dev())
    N.grouped_gemm_nvfp4_fwd_rht_s2f6(hq.sg, hq.codes, hq.scales, wq.codes, wq.scales, wq.sg, go, E, M, N_, K, mask,
                                      y, c, s)
    check_status()
    assert torch.equal(c, c_ref) and torch.equal(s, s_ref)
    if with_y:
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))


def M_seed(sizes):
    return int(sum(sizes)) + len(sizes)


@pytest.mark.parametrize("with_y", [True, False])
@pytest.mark.parametrize("sizes,N_,K,mask", [([37, 0, 200, 128], 256, 512, 0x9E3779B9), ([300, 1], 128, 256, 0)])
def test_w2_epilogue_rht_s2f6_equals_gemm_then_quantize(sizes, N_, K, mask, with_y):
    """The w2 GEMM's RHT + S2F6 epilogue: codes and scales identical to the
    plain bf16 GEMM followed by rht32_s2f6_quantize (and the bf16 output, when
    requested, identical to the plain GEMM's)."""
    _fused_vs_separate(sizes, N_, K, mask, with_y)


def test_w2_epilogue_rht_s2f6_full_size():
    """The MoE layer's w2 GEMM at full size (131072 routed rows, d_ff 1536 ->
    d_model 4096, 64 uneven experts): fused == separate over every element."""
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    m = W.moe("cpu", seed=2, tokens=16384, weights=False)
    sizes = np.diff(m.group_offsets.numpy()).tolist()
    _fused_vs_separate(sizes, 4096, 1536, 0x6A09E667, with_y=False)
