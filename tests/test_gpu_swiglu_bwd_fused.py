"""grouped_gemm_mxfp8_dx_swiglu_bwd against the unfused sequence, bit for bit:
dh = grouped_gemm_mxfp8_dx (bf16 output), then dy13 = nvfp4moe_swiglu_bwd(dh,
y13); every kernel choice, ragged and empty groups, several hidden widths;
rows past the last routed row and the other half of each row are left
untouched; and a whole MoE step with and without the fused epilogue gives
identical outputs."""
import numpy as np
import pytest
import torch

from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
from precision_moe_numerics_nvfp4_gb300 import pipeline as PL
from precision_moe_numerics_nvfp4_gb300 import workloads as W
from precision_moe_numerics_nvfp4_gb300.pipeline import MxRows, MxTransposed, NvTensor
from tests.gpu_helpers import check_status, dev, gfull

pytestmark = pytest.mark.gpu


def _rand(shape, seed, std):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * std).to(torch.bfloat16).contiguous()


@pytest.fixture(params=[N.GEMM_AUTO, N.GEMM_ONE_PER_SM, N.GEMM_TWO_PER_SM, N.GEMM_CTA_PAIR, N.GEMM_CTA_PAIR_N128],
                ids=["auto", "one_per_sm", "two_per_sm", "cta_pair", "cta_pair_n128"])
def gemm_kernel(request):
    """The fused epilogue exists in every dgrad kernel; each must match the
    unfused sequence run with the same kernel choice."""
    N.nvfp4moe_set_gemm_kernel(request.param)
    yield request.param
    N.nvfp4moe_set_gemm_kernel(N.GEMM_AUTO)


def _operands(sizes, Nd, I, seed):
    """g [M, Nd] -> MXFP8 SR row-wise; w2 [E, Nd, I] -> NVFP4 -> requant
    transposed [E][I][Nd]; y13 [M, 2I] bf16."""
    o = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    go = torch.from_numpy(o).to(dev())
    M, E = int(o[-1]), len(sizes)
    g = _rand((M, Nd), seed, 1e-3)
    w = _rand((E, Nd, I), seed + 1, 0.02)
    y13 = _rand((M, 2 * I), seed + 2, 1.0)
    wq = NvTensor(E, Nd, I, dev())
    wq.quantize(w)
    wt = MxTransposed(Nd, I, dev(), batch=E)
    N.dequant_transpose_requant_sr(wq.codes, wq.scales, wq.sg, E, Nd, I, None, 3, 0, wt.codes, wt.scales)
    gr, gt = MxRows(M, Nd, dev(), E=E), MxTransposed(M, Nd, dev(), E=E)
    N.mxfp8_quantize(g, M, Nd, go, N.NV_SR, 3, 4, 5, gr.codes, gr.scales, gt.codes, gt.scales)
    check_status()
    return go, M, E, gr, wt, y13


@pytest.mark.parametrize("sizes,Nd,I", [([300], 256, 128), ([5, 0, 295, 130, 1], 512, 256), ([0, 700, 0], 256, 384),
                                        ([128, 128], 1024, 1536), ([600, 1, 0, 257, 513], 512, 256)])
def test_fused_swiglu_bwd_equals_unfused(sizes, Nd, I, gemm_kernel):
    go, M, E, gr, wt, y13 = _operands(sizes, Nd, I, seed=Nd + I + len(sizes))
    dh = gfull((M, I), 7, dtype=torch.bfloat16, device=dev())
    ref = gfull((M + 3, 2 * I), 7, dtype=torch.bfloat16, device=dev())
    N.grouped_gemm_mxfp8_dx(gr.codes, gr.scales, wt.codes, wt.scales, go, E, M, Nd, I, dh, N.NV_OUT_BF16)
    N.nvfp4moe_swiglu_bwd(dh, y13, M, I, ref)
    out = gfull((M + 3, 2 * I), 7, dtype=torch.bfloat16, device=dev())  # 3 rows past the end stay untouched
    N.grouped_gemm_mxfp8_dx_swiglu_bwd(gr.codes, gr.scales, wt.codes, wt.scales, go, E, M, Nd, I, y13, out)
    check_status()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.all(out[M:] == 7)


def test_fused_swiglu_bwd_rejects_overlap_and_bad_shapes():
    go, M, E, gr, wt, y13 = _operands([64, 64], 256, 128, seed=5)
    f = N.lib().grouped_gemm_mxfp8_dx_swiglu_bwd
    P = N._ptr
    args = (P(gr.codes), P(gr.scales), P(wt.codes), P(wt.scales), P(go), E, M, 256)
    assert f(*args, 128, P(y13), P(y13), None) == N.NV_ERR_ARG          # in place
    assert f(*args, 192, P(y13), P(gfull((M, 384), 0, dtype=torch.bfloat16, device=dev())), None) == N.NV_ERR_SHAPE
    assert f(*args, 128, None, P(y13), None) == N.NV_ERR_ARG


def test_moe_step_with_and_without_fused_swiglu_bwd():
    """A small MoE step: every output of the fused backward equals the unfused
    one (dh stored, then nvfp4moe_swiglu_bwd)."""
    m = W.moe("cuda", seed=5, tokens=512, d_model=256, experts=6, topk=2, d_ff=256, with_grad=True, grad_seed=3)
    M = m.x_perm.shape[0]
    outs = []
    for fused in (True, False):
        layer = PL.MoELayer(M, 256, 256, 6, fuse_swiglu_bwd=fused)
        assert layer.fuse_swiglu_bwd == fused and (layer.dh is None) == fused
        layer.step(m.x_perm, m.w13, m.w2, m.g2, m.group_offsets, seed=3)
        check_status()
        outs.append([t.clone() for t in (layer.y2, layer.dy13, layer.dx, layer.dw2, layer.dw13)])
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b)
