"""Four Over Six on the GPU against the oracle's reading of it ("Recipe
details": two candidate block scales for activations; the selection rule is a
reading, see the oracle): codes, scales and outer scales bit-exact for
batched and grouped inputs, blocks that each mapping represents exactly,
zero blocks, the fused quantize + SR re-quantization equal to the two calls,
and sampled rows of the full-size activation."""
import numpy as np
import pytest
import torch

from oracle import layout as L
from oracle import nvfp4 as NV
from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
from precision_moe_numerics_nvfp4_gb300.pipeline import MxTransposed, NvTensor
from tests.gpu_helpers import bf16_f32, check_status, dev

pytestmark = pytest.mark.gpu


def _x(shape, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn(shape, generator=g, device="cuda")
    flat = x.view(-1)
    idx = torch.randperm(flat.numel(), generator=g, device="cuda")[: max(1, flat.numel() // 3000)]
    flat[idx] *= 50.0
    return x.to(torch.bfloat16).contiguous()


def _expected(xf, batch, rows, cols, o=None, sg_in=None):
    codes, logical, sgs = [], [], []
    xb = xf.reshape(batch, rows, cols)
    for b in range(batch):
        c, s, sg = NV.quantize_four_over_six(xb[b], None if sg_in is None else np.float32(sg_in[b]))
        codes.append(NV.pack(c))
        logical.append(s)
        sgs.append(sg)
    if o is None:
        buf = L.swizzle(np.concatenate(logical), L.batched_row_map(batch, rows), batch * L.roundup(rows, 128))
    else:
        buf = L.swizzle(np.concatenate(logical), L.grouped_row_map(o), L.padded_cap(rows, len(o) - 1))
    return np.concatenate(codes).reshape(-1), buf, np.array(sgs, np.float32)


def _gpu(x, batch, rows, cols, go=None, sg_in=None):
    E = None if go is None else go.numel() - 1
    t = NvTensor(batch, rows, cols, dev(), E=E)
    t.codes.fill_(0xA5)
    t.scales.fill_(0xA5)
    N.nvfp4_quantize_four_over_six(x, batch, rows, cols, go, sg_in, t.sg, t.codes, t.scales,
                                   None if sg_in is not None else t.ws)
    check_status()
    return t


@pytest.mark.parametrize("batch,rows,cols", [(1, 128, 128), (3, 200, 256), (2, 384, 1024)])
def test_batched_matches_oracle(batch, rows, cols):
    x = _x((batch, rows, cols), seed=batch * 7 + rows)
    t = _gpu(x, batch, rows, cols)
    ec, es, esg = _expected(bf16_f32(x), batch, rows, cols)
    assert np.array_equal(t.sg.cpu().numpy(), esg)
    assert np.array_equal(t.codes.cpu().numpy()[: ec.size], ec)
    assert np.array_equal(t.scales.cpu().numpy(), es)


@pytest.mark.parametrize("sizes,cols", [([5, 0, 295, 130, 1], 512), ([0, 700], 128)])
def test_grouped_matches_oracle(sizes, cols):
    o = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    go = torch.from_numpy(o).to(dev())
    rows = int(o[-1])
    x = _x((rows, cols), seed=rows + cols)
    t = _gpu(x, 1, rows, cols, go)
    ec, es, esg = _expected(bf16_f32(x), 1, rows, cols, o.astype(np.int64))
    assert np.array_equal(t.sg.cpu().numpy(), esg)
    assert np.array_equal(t.codes.cpu().numpy()[: ec.size], ec)
    assert np.array_equal(t.scales.cpu().numpy(), es)


def test_exact_blocks_and_zero_blocks_with_given_outer_scale():
    b4 = [4, 3, 2, 1.5, 1, 0.5, 0, -4, -3, -2, -1.5, -1, -0.5, 0, 3, 2]
    b6 = [6, 4, 3, 2, 1.5, 1, 0.5, 0, -6, -4, -3, -2, -1.5, -1, -0.5, 0]
    rows = np.zeros((128, 128), np.float32)
    rows[0, :16], rows[0, 16:32], rows[1, :16] = b4, b6, b6
    rows[1, 16:32] = b4
    x = torch.from_numpy(rows).to(torch.bfloat16).to(dev())
    sg_in = torch.ones(1, dtype=torch.float32, device=dev())
    t = _gpu(x, 1, 128, 128, sg_in=sg_in)
    ec, es, _ = _expected(bf16_f32(x), 1, 128, 128, sg_in=np.ones(1, np.float32))
    assert np.array_equal(t.codes.cpu().numpy()[: ec.size], ec)
    assert np.array_equal(t.scales.cpu().numpy(), es)
    s = L.unswizzle(t.scales.cpu().numpy(), L.batched_row_map(1, 128), 8)
    assert s[0, 0] == 0x38 and s[0, 1] == 0x38 and s[1, 0] == 0x38   # E4M3 1.0: both exact blocks keep scale 1


@pytest.mark.parametrize("sizes,cols", [([5, 0, 295, 130, 1], 256), ([256], 512)])
def test_fused_requant_equals_separate(sizes, cols):
    o = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    go = torch.from_numpy(o).to(dev())
    rows, E = int(o[-1]), len(sizes)
    x = _x((rows, cols), seed=rows * 3)
    a = _gpu(x, 1, rows, cols, go)
    ma = MxTransposed(rows, cols, dev(), E=E)
    mb = MxTransposed(rows, cols, dev(), E=E)
    for t in (ma.codes, ma.scales, mb.codes, mb.scales):
        t.fill_(0x5A)
    N.dequant_transpose_requant_sr(a.codes, a.scales, a.sg, 1, rows, cols, go, 5, 2, ma.codes, ma.scales)
    b = NvTensor(1, rows, cols, dev(), E=E)
    N.nvfp4_quantize_requant_four_over_six(x, 1, rows, cols, go, None, b.sg, b.codes, b.scales, b.ws, 5, 2,
                                           mb.codes, mb.scales)
    check_status()
    assert torch.equal(a.sg, b.sg) and torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
    assert torch.equal(ma.codes, mb.codes) and torch.equal(ma.scales, mb.scales)


def test_full_size_sampled_rows():
    """The MoE activation (131072 routed rows x 4096, 64 uneven groups): 48
    sampled rows bit-exact against the oracle."""
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    m = W.moe("cuda", seed=2, tokens=16384, weights=False)
    x, go = m.x_perm, m.group_offsets
    rows, cols = x.shape
    t = _gpu(x, 1, rows, cols, go)
    sg = t.sg.cpu().numpy()[0]
    pick = torch.randint(0, rows, (48,), generator=torch.Generator().manual_seed(3)).numpy()
    xs = bf16_f32(x[torch.from_numpy(pick).to(dev())])
    assert sg == NV.outer_scale(bf16_f32(x))
    c, s, _ = NV.quantize_four_over_six(xs, sg)
    assert np.array_equal(t.codes.view(rows, cols // 2).cpu().numpy()[pick], NV.pack(c))
    full = L.unswizzle(t.scales.cpu().numpy(), L.grouped_row_map(go.cpu().numpy().astype(np.int64)), cols // 16)
    assert np.array_equal(full[pick], s)
