"""Per-token activation outer scales on the GPU against the oracle
("Recipe details": one FP32 scale per token).  Codes, scales and per-row
outer scales bit-exact (grouped with ragged and empty groups, and plain); the
fused quantize + SR re-quantization equal to the two separate calls bit for
bit and to the oracle's per-row re-quantization; batch invariance; the
forward GEMM with per-row scales within 1e-4 (|A||B|) of the FP64 product of
the dequantized operands; the SwiGLU epilogue's per-row outer scales of h
equal to the per-row rule applied to h; bad arguments rejected; and sampled
rows of the full-size activation."""
import numpy as np
import pytest
import torch

from oracle import gemm as G
from oracle import layout as L
from oracle import nvfp4 as NV
from oracle import requant as RQ
from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
from precision_moe_numerics_nvfp4_gb300.pipeline import MxTransposed, NvTensor
from tests.gpu_helpers import bf16_f32, check_status, dev, filled, gempty, gfull, unpack_gpu_nvfp4

pytestmark = pytest.mark.gpu


def _x(rows, cols, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    # tokens of very different magnitudes: what per-token scales are for
    mag = torch.exp(gempty((rows, 1), device="cuda").uniform_(-8, 8, generator=g))
    x = torch.randn((rows, cols), generator=g, device="cuda") * mag
    if rows > 4:
        x[2] = 0.0                      # an all-zero token
        x[3, 5] = 1e4                   # an outlier inside a token
    return x.to(torch.bfloat16).contiguous()


def _groups(sizes):
    o = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    return torch.from_numpy(o).to(dev()), o.astype(np.int64)


def _expected(xf, o):
    c, s, sg = NV.quantize_rows(xf)
    rmap = L.batched_row_map(1, xf.shape[0]) if o is None else L.grouped_row_map(o)
    prow = L.roundup(xf.shape[0], 128) if o is None else L.padded_cap(xf.shape[0], len(o) - 1)
    return NV.pack(c).reshape(-1), L.swizzle(s, rmap, prow), sg, c, s


def _gpu_rows(x, rows, cols, go, E):
    t = NvTensor(1, rows, cols, dev(), E=E)
    t.codes.fill_(0xA5)
    t.scales.fill_(0xA5)
    sg = gfull((rows,), -1.0, dtype=torch.float32, device=dev())
    N.nvfp4_quantize_rows(x, rows, cols, go, None, sg, t.codes, t.scales)
    check_status()
    return t, sg


@pytest.mark.parametrize("sizes,cols", [(None, 256), ([5, 0, 295, 130, 1], 512), ([0, 0, 700], 128),
                                        ([129, 127, 128, 0], 1536)])
def test_quantize_rows_matches_oracle(sizes, cols):
    go, o = (None, None) if sizes is None else _groups(sizes)
    rows = 300 if sizes is None else int(o[-1])
    x = _x(rows, cols, seed=rows + cols)
    t, sg = _gpu_rows(x, rows, cols, go, None if sizes is None else len(sizes))
    ec, es, esg, _, _ = _expected(bf16_f32(x), o)
    assert np.array_equal(sg.cpu().numpy(), esg)
    assert np.array_equal(t.codes.cpu().numpy()[: ec.size], ec)
    assert np.array_equal(t.scales.cpu().numpy(), es)


def test_given_row_scales_are_used_and_copied():
    rows, cols = 256, 256
    x = _x(rows, cols, seed=3)
    sg_in = torch.exp(torch.linspace(-3, 3, rows, device=dev())).float()
    t = NvTensor(1, rows, cols, dev())
    out = torch.zeros(rows, dtype=torch.float32, device=dev())
    N.nvfp4_quantize_rows(x, rows, cols, None, sg_in, out, t.codes, t.scales)
    check_status()
    c, s, _ = NV.quantize_rows(bf16_f32(x), sg_in.cpu().numpy())
    assert torch.equal(out, sg_in)
    assert np.array_equal(t.codes.cpu().numpy()[: rows * cols // 2], NV.pack(c).reshape(-1))
    assert np.array_equal(L.unswizzle(t.scales.cpu().numpy(), L.batched_row_map(1, rows), cols // 16), s)


def test_batch_invariance_on_the_gpu():
    rows, cols = 384, 512
    x = _x(rows, cols, seed=5)
    y = x.clone()
    y[100] = y[100] * 1000
    a, _ = _gpu_rows(x, rows, cols, None, None)
    b, _ = _gpu_rows(y, rows, cols, None, None)
    ca = a.codes.view(rows, cols // 2)
    cb = b.codes.view(rows, cols // 2)
    keep = torch.arange(rows, device=dev()) != 100
    assert torch.equal(ca[keep], cb[keep])
    sa = L.unswizzle(a.scales.cpu().numpy(), L.batched_row_map(1, rows), cols // 16)
    sb = L.unswizzle(b.scales.cpu().numpy(), L.batched_row_map(1, rows), cols // 16)
    k = keep.cpu().numpy()
    assert np.array_equal(sa[k], sb[k])


@pytest.mark.parametrize("sizes,cols", [([5, 0, 295, 130, 1], 256), ([256], 512), ([1, 130, 0, 3], 128)])
def test_quantize_requant_rows_fused_separate_and_oracle(sizes, cols):
    go, o = _groups(sizes)
    rows, E = int(o[-1]), len(sizes)
    x = _x(rows, cols, seed=rows + 17)
    a, sga = _gpu_rows(x, rows, cols, go, E)
    ma = MxTransposed(rows, cols, dev(), E=E)
    for t in (ma.codes, ma.scales):  # same fill as the fused call's buffers (columns past the groups stay unwritten)
        t.fill_(0x5A)
    N.dequant_transpose_requant_sr_rows(a.codes, a.scales, sga, rows, cols, go, 7, 2, ma.codes, ma.scales)
    b = NvTensor(1, rows, cols, dev(), E=E)
    mb = MxTransposed(rows, cols, dev(), E=E)
    for t in (b.codes, b.scales, mb.codes, mb.scales):
        t.fill_(0x5A)
    sgb = gempty(rows, dtype=torch.float32, device=dev())
    N.nvfp4_quantize_requant_rows(x, rows, cols, go, None, sgb, b.codes, b.scales, 7, 2, mb.codes, mb.scales)
    check_status()
    assert torch.equal(sga, sgb) and torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
    assert torch.equal(ma.codes, mb.codes) and torch.equal(ma.scales, mb.scales)
    c, s = unpack_gpu_nvfp4(b.codes.cpu().numpy(), b.scales.cpu().numpy(), 1, rows, cols, o)
    P = N.nvfp4moe_padded_cap(rows, E)
    ec, es = RQ.requant_grouped_rows(c, s, sgb.cpu().numpy(), o, 7, 2, P)
    Ptot = int(L.group_padded_starts(o)[-1])
    assert np.array_equal(mb.codes.cpu().numpy().reshape(cols, P)[:, :Ptot], ec[:, :Ptot])
    assert np.array_equal(L.unswizzle(mb.scales.cpu().numpy(), np.arange(cols), P // 32), es)


def _weights(E, n, k, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    w = (torch.randn((E, n, k), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    wq = NvTensor(E, n, k, dev())
    wq.quantize(w)
    return wq


@pytest.fixture(params=[N.GEMM_AUTO, N.GEMM_CTA_PAIR], ids=["auto", "cta_pair"])
def gemm_kernel(request):
    """Per-token outer scales in the 128 x 128 kernel's epilogue and in the
    CTA-pair kernel's (shapes whose width is not a multiple of 256 fall back
    to the former)."""
    N.nvfp4moe_set_gemm_kernel(request.param)
    yield request.param
    N.nvfp4moe_set_gemm_kernel(N.GEMM_AUTO)


@pytest.mark.parametrize("sizes,N_,K", [([37, 0, 200, 128], 256, 512), ([300, 1], 128, 256)])
def test_fwd_gemm_rows_within_bound(sizes, N_, K, gemm_kernel):
    go, o = _groups(sizes)
    M, E = int(o[-1]), len(sizes)
    x = _x(M, K, seed=M + K)
    xq, sgx = _gpu_rows(x, M, K, go, E)
    wq = _weights(E, N_, K, seed=E)
    y = gempty((M, N_), dtype=torch.float32, device=dev())
    N.grouped_gemm_nvfp4_fwd_rows(sgx, xq.codes, xq.scales, wq.codes, wq.scales, wq.sg, go, E, M, N_, K, y,
                                  N.NV_OUT_FP32)
    check_status()
    c, s = unpack_gpu_nvfp4(xq.codes.cpu().numpy(), xq.scales.cpu().numpy(), 1, M, K, o)
    A64 = NV.dequantize_rows_f64(c, s, sgx.cpu().numpy())
    wc, ws = unpack_gpu_nvfp4(wq.codes.cpu().numpy(), wq.scales.cpu().numpy(), E, N_, K)
    B64 = np.stack([NV.dequantize_f64(wc.reshape(E, N_, K)[e], ws.reshape(E, N_, K // 16)[e],
                                      wq.sg.cpu().numpy()[e]) for e in range(E)])
    ref, bound = G.grouped_rows(A64, B64, o)
    assert G.within_bound(y.cpu().numpy(), ref, bound).all()


def test_swiglu_rows_epilogue(gemm_kernel):
    sizes, I, K = [40, 0, 300, 129], 128, 512
    go, o = _groups(sizes)
    M, E = int(o[-1]), len(sizes)
    x = _x(M, K, seed=77)
    xq, sgx = _gpu_rows(x, M, K, go, E)
    wq = _weights(E, 2 * I, K, seed=8)
    y13 = gempty((M, 2 * I), dtype=torch.bfloat16, device=dev())
    h = gempty((M, I), dtype=torch.bfloat16, device=dev())
    hsg = gfull((M,), -1.0, dtype=torch.float32, device=dev())
    N.grouped_gemm_nvfp4_fwd_swiglu_rows(sgx, xq.codes, xq.scales, wq.codes, wq.scales, wq.sg, go, E, M, I, K,
                                         y13, h, hsg)
    y_ref = torch.empty_like(y13)
    N.grouped_gemm_nvfp4_fwd_rows(sgx, xq.codes, xq.scales, wq.codes, wq.scales, wq.sg, go, E, M, 2 * I, K, y_ref,
                                  N.NV_OUT_BF16)
    h_ref = torch.empty_like(h)
    N.nvfp4moe_swiglu_fwd(y_ref, M, I, h_ref)
    check_status()
    assert torch.equal(y13.view(torch.int16), y_ref.view(torch.int16))
    assert torch.equal(h.view(torch.int16), h_ref.view(torch.int16))
    assert np.array_equal(hsg.cpu().numpy(), NV.outer_scale_rows(bf16_f32(h)))


def test_rows_rejects_bad_arguments():
    x = torch.zeros((128, 128), dtype=torch.bfloat16, device=dev())
    t = NvTensor(1, 128, 128, dev())
    with pytest.raises(N.NvError):
        N.nvfp4_quantize_rows(x, 128, 128, None, None, None, t.codes, t.scales)   # no scale in or out
    sg = torch.zeros(129, dtype=torch.float32, device=dev())
    with pytest.raises(N.NvError):
        N.nvfp4_quantize_rows(x, 128, 120, None, None, sg, t.codes, t.scales)     # cols % 16
    with pytest.raises(N.NvError):
        N.nvfp4_quantize_rows(x, 128, 128, None, None, sg.view(torch.uint8)[1:], t.codes, t.scales)  # misaligned
    check_status()


def test_full_size_sampled_rows():
    """The MoE activation: 16384 tokens x top-8 = 131072 routed rows x 4096 in
    64 uneven groups, quantized with per-token scales and re-quantized in the
    launch the training step makes; 64 sampled rows bit-exact (codes, block
    scales, outer scales) against the oracle."""
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    m = W.moe("cuda", seed=2, tokens=16384, weights=False)
    x, go = m.x_perm, m.group_offsets
    rows, cols, E = x.shape[0], x.shape[1], go.numel() - 1
    t = NvTensor(1, rows, cols, dev(), E=E)
    mx = MxTransposed(rows, cols, dev(), E=E)
    sg = gempty(rows, dtype=torch.float32, device=dev())
    N.nvfp4_quantize_requant_rows(x, rows, cols, go, None, sg, t.codes, t.scales, 3, 2, mx.codes, mx.scales)
    check_status()
    pick = torch.randint(0, rows, (64,), generator=torch.Generator().manual_seed(1))
    xs = bf16_f32(x[pick.to(dev())])
    c, s, esg = NV.quantize_rows(xs)
    assert np.array_equal(sg.cpu().numpy()[pick.numpy()], esg)
    codes = t.codes.view(rows, cols // 2).cpu().numpy()[pick.numpy()]
    assert np.array_equal(codes, NV.pack(c))
    o = go.cpu().numpy().astype(np.int64)
    full = L.unswizzle(t.scales.cpu().numpy(), L.grouped_row_map(o), cols // 16)
    assert np.array_equal(full[pick.numpy()], s)


def test_moe_layer_per_token_variants_agree():
    """The per-token MoE layer: the fused (SwiGLU epilogue, quantize +
    re-quantize) and unfused paths give the same forward and backward outputs
    bit for bit; x and h carry the per-row rule's scales and codes."""
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    from precision_moe_numerics_nvfp4_gb300.pipeline import MoELayer
    m = W.moe("cuda", seed=2, tokens=160, d_model=256, experts=8, topk=4, d_ff=256, with_grad=True)
    M, d, I, E = m.x_perm.shape[0], 256, 256, 8
    outs = []
    for fs, fr in [(True, True), (False, True), (True, False), (False, False)]:
        layer = MoELayer(M, d, I, E, fuse_swiglu=fs, fuse_requant=fr, per_token=True)
        layer.forward(m.x_perm, m.w13, m.w2, m.group_offsets, seed=3)
        layer.backward(m.g2, m.group_offsets, seed=3)
        check_status()
        o = m.group_offsets.cpu().numpy().astype(np.int64)
        Ptot = int(L.group_padded_starts(o)[-1])
        P = N.nvfp4moe_padded_cap(M, E)
        # written regions only (the transposed operands leave the columns past
        # the last group's padding untouched)
        outs.append([t.clone() for t in (layer.x_sg_rows, layer.h_sg_rows, layer.xq.codes[: M * d // 2],
                                         layer.hq.codes[: M * I // 2], layer.y2, layer.dx, layer.dw13, layer.dw2,
                                         layer.xt.codes[: d * P].view(d, P)[:, :Ptot],
                                         layer.ht.codes[: I * P].view(I, P)[:, :Ptot])])
        if fs and fr:
            xs = bf16_f32(m.x_perm)
            assert np.array_equal(layer.x_sg_rows.cpu().numpy(), NV.outer_scale_rows(xs))
            assert np.array_equal(layer.h_sg_rows.cpu().numpy(), NV.outer_scale_rows(bf16_f32(layer.h)))
            c, _, _ = NV.quantize_rows(xs)
            assert np.array_equal(layer.xq.codes.cpu().numpy()[: M * d // 2], NV.pack(c).reshape(-1))
    for other in outs[1:]:
        for i, (a, b) in enumerate(zip(outs[0], other)):
            assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8)), i
