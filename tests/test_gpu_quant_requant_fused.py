"""nvfp4_quantize_requant must equal nvfp4_quantize followed by
dequant_transpose_requant_sr bit for bit (codes, scales, outer scales and the
MXFP8 codes and scales), for batched weights and grouped activations with
ragged and empty groups, with the outer scale computed or given; and one case
is checked against the oracle directly."""
import numpy as np
import pytest
import torch

from oracle import layout as L
from oracle import requant as RQ
from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
from precision_moe_numerics_nvfp4_gb300.pipeline import MxTransposed, NvTensor
from tests.gpu_helpers import check_status, dev, oracle_nvfp4

pytestmark = pytest.mark.gpu


def _x(shape, seed, std=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn(shape, generator=g, device="cuda") * std
    flat = x.view(-1)
    idx = torch.randperm(flat.numel(), generator=g, device="cuda")[: max(1, flat.numel() // 5000)]
    flat[idx] *= 300.0  # outliers: wide-range blocks
    return x.to(torch.bfloat16).contiguous()


def _both(x, batch, rows, cols, groups, sg_in, seed, off):
    E = None if groups is None else groups.numel() - 1
    a, b = NvTensor(batch, rows, cols, dev(), E=E), NvTensor(batch, rows, cols, dev(), E=E)
    if groups is None:
        ma, mb = MxTransposed(rows, cols, dev(), batch=batch), MxTransposed(rows, cols, dev(), batch=batch)
    else:
        ma, mb = MxTransposed(rows, cols, dev(), E=E), MxTransposed(rows, cols, dev(), E=E)
    for t in (a.codes, a.scales, b.codes, b.scales, ma.codes, ma.scales, mb.codes, mb.scales):
        t.fill_(0xA5)
    N.nvfp4_quantize(x, batch, rows, cols, groups, sg_in, a.sg, a.codes, a.scales, a.ws)
    N.dequant_transpose_requant_sr(a.codes, a.scales, a.sg, batch, rows, cols, groups, seed, off, ma.codes, ma.scales)
    N.nvfp4_quantize_requant(x, batch, rows, cols, groups, sg_in, b.sg, b.codes, b.scales, b.ws, seed, off,
                             mb.codes, mb.scales)
    check_status()
    return (a, ma), (b, mb)


def _assert_same(sep, fused):
    (a, ma), (b, mb) = sep, fused
    assert torch.equal(a.sg, b.sg)
    assert torch.equal(a.codes, b.codes)
    assert torch.equal(a.scales, b.scales)
    assert torch.equal(ma.codes, mb.codes)
    assert torch.equal(ma.scales, mb.scales)


@pytest.mark.parametrize("batch,rows,cols", [(1, 128, 128), (3, 256, 384), (4, 384, 1024)])
def test_fused_equals_separate_batched(batch, rows, cols):
    x = _x((batch, rows, cols), seed=batch + rows, std=0.02)
    _assert_same(*_both(x, batch, rows, cols, None, None, seed=7, off=1))


@pytest.mark.parametrize("sizes,cols", [([300], 256), ([5, 0, 295, 130, 1], 512), ([0, 0, 700], 128),
                                        ([129, 127, 128, 0], 1536)])
def test_fused_equals_separate_grouped(sizes, cols):
    o = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    groups = torch.from_numpy(o).to(dev())
    M = int(o[-1])
    x = _x((M, cols), seed=M + cols)
    _assert_same(*_both(x, 1, M, cols, groups, None, seed=3, off=2))


def test_fused_with_given_outer_scale():
    x = _x((2, 128, 256), seed=9)
    sg = torch.tensor([0.5, 3.0], dtype=torch.float32, device=dev())
    _assert_same(*_both(x, 2, 128, 256, None, sg, seed=1, off=0))


@pytest.mark.parametrize("sg", [1.0, 1e-39], ids=["table_range", "below_table_range"])
def test_fused_subnormal_block_maxima(sg):
    """Blocks of bf16 subnormals (|x| < 2^-126, some zero) beside normal
    blocks: under an outer scale whose 6 sg lies in the block-scale table's
    range the fused kernel reads the subnormal quotients from the table, under
    a tiny one it divides; both must match the separate quantizer."""
    rows, cols = 128, 256
    g = torch.Generator(device="cuda").manual_seed(31)
    x = torch.randn((1, rows, cols), generator=g, device="cuda") * 0.5
    x[:, :, :64] *= 2.0 ** -130
    x[:, ::3, 64:96] *= 2.0 ** -136
    x = x.to(torch.bfloat16).contiguous()
    assert (x[:, :, :64].float().abs().max() < 2.0 ** -126).item()
    sg_in = torch.tensor([sg], dtype=torch.float32, device=dev())
    _assert_same(*_both(x, 1, rows, cols, None, sg_in, seed=4, off=3))


def test_fused_against_oracle():
    batch, rows, cols, seed, off = 2, 128, 256, 11, 5
    x = _x((batch, rows, cols), seed=21, std=0.02)
    (_, _), (b, mb) = _both(x, batch, rows, cols, None, None, seed, off)
    codes, scales, sg = oracle_nvfp4(x.float().cpu().numpy(), batch, rows, cols)
    assert np.array_equal(b.codes.cpu().numpy()[: codes.size], codes)
    assert np.array_equal(b.sg.cpu().numpy(), sg)
    from oracle import nvfp4 as NV
    lc = NV.unpack(codes.reshape(batch * rows, cols // 2))
    ls = L.unswizzle(scales, L.batched_row_map(batch, rows), cols // 16)
    want_c, want_s = RQ.requant_weights(lc.reshape(batch, rows, cols), ls.reshape(batch, rows, cols // 16), sg,
                                        seed, off)
    got_c = mb.codes.cpu().numpy()[: want_c.size].reshape(want_c.shape)
    assert np.array_equal(got_c, want_c)
    got_s = L.unswizzle(mb.scales.cpu().numpy(), L.batched_row_map(batch, cols), rows // 32)
    assert np.array_equal(got_s.reshape(want_s.shape), want_s)


def test_outer_scale_alone_equals_quantize_and_feeds_back():
    """nvfp4_outer_scale computes the outer scales nvfp4_quantize computes;
    given back as outer_scale_in they reproduce its result bit for bit."""
    batch, rows, cols = 3, 256, 384
    x = _x((batch, rows, cols), seed=77, std=0.05)
    a = NvTensor(batch, rows, cols, dev())
    N.nvfp4_quantize(x, batch, rows, cols, None, None, a.sg, a.codes, a.scales, a.ws)
    b = NvTensor(batch, rows, cols, dev())
    N.nvfp4_outer_scale(x, batch, rows * cols, b.sg, b.ws)
    N.nvfp4_quantize(x, batch, rows, cols, None, b.sg, b.sg, b.codes, b.scales, None)
    check_status()
    assert torch.equal(a.sg, b.sg) and torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)


def test_moe_layer_side_stream_amax_equals_inline():
    """The layer's side-stream amax passes change nothing: forward and
    backward outputs equal the inline-amax layer's bit for bit."""
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    from precision_moe_numerics_nvfp4_gb300.pipeline import MoELayer
    m = W.moe("cuda", seed=2, tokens=160, d_model=256, experts=8, topk=4, d_ff=256, with_grad=True)
    M = m.x_perm.shape[0]
    outs = []
    for overlap in (True, False):
        layer = MoELayer(M, 256, 256, 8, overlap_amax=overlap)
        for _ in range(2):  # a second step reuses the scale buffers
            layer.step(m.x_perm, m.w13, m.w2, m.g2, m.group_offsets, seed=3)
        torch.cuda.synchronize()
        check_status()
        outs.append([t.clone() for t in (layer.xq.sg, layer.w13q.sg, layer.w2q.sg, layer.y2, layer.dx, layer.dw13,
                                         layer.dw2)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)
