"""GPU parity of the grouped GEMMs (NVFP4 forward, MXFP8 dgrad and wgrad)
against the FP64 oracle:
every output element within 1e-4 * (|A||B|)_ij of the exact product of the
dequantized operands (plus half a bf16 ulp for bf16 outputs).  The operands
are the GPU's own quantized tensors, whose bit-exactness the quantizer tests
establish; the oracle dequantizes them independently."""
import numpy as np
import pytest
import torch

from oracle import gemm as G
from oracle import layout as L
from oracle import mxfp8 as MX
from oracle import nvfp4 as NV
from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
from precision_moe_numerics_nvfp4_gb300 import workloads as W
from precision_moe_numerics_nvfp4_gb300.pipeline import MxRows, MxTransposed, NvTensor, SingleLinear
from tests.gpu_helpers import bf16_f32, check_status, dev, gempty, gfull, unpack_gpu_nvfp4

pytestmark = pytest.mark.gpu


def _rand(shape, seed, std=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * std).to(torch.bfloat16).contiguous()


def _groups(sizes):
    o = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    return torch.from_numpy(o).to(dev()), o


def _deq_nvfp4(t: NvTensor, groups=None):
    c, s = unpack_gpu_nvfp4(t.codes.cpu().numpy(), t.scales.cpu().numpy(), t.batch, t.rows, t.cols, groups)
    sg = t.sg.cpu().numpy()
    if t.batch == 1:
        return NV.dequantize_f64(c, s, sg[0])
    rows = t.rows
    return np.stack([NV.dequantize_f64(c[b * rows:(b + 1) * rows], s[b * rows:(b + 1) * rows], sg[b])
                     for b in range(t.batch)])


def _fwd(sizes, N_, K, out_fp32=True, seed=0):
    go, o = _groups(sizes)
    M, E = int(o[-1]), len(sizes)
    x = _rand((M, K), seed)
    w = _rand((E, N_, K), seed + 1, 0.02)
    xq, wq = NvTensor(1, M, K, dev(), E=E), NvTensor(E, N_, K, dev())
    xq.quantize(x, go)
    wq.quantize(w)
    y = gfull((M, N_), float("nan"), dtype=torch.float32 if out_fp32 else torch.bfloat16, device=dev())
    N.grouped_gemm_nvfp4_fwd(None, xq.sg, xq.codes, xq.scales, wq.codes, wq.scales, wq.sg, go, E, M, N_, K, y,
                             N.NV_OUT_FP32 if out_fp32 else N.NV_OUT_BF16)
    check_status()
    return y, xq, wq, o


@pytest.fixture(params=[N.GEMM_TWO_PER_SM, N.GEMM_CTA_PAIR, N.GEMM_ONE_PER_SM, N.GEMM_CTA_PAIR_N128],
                ids=["two_per_sm", "cta_pair", "one_per_sm", "cta_pair_n128"])
def gemm_kernel(request):
    """Each kernel choice must meet the same bound; shapes whose output width
    is not a multiple of 256 run the 128 x 128 kernel under every choice."""
    N.nvfp4moe_set_gemm_kernel(request.param)
    yield request.param
    N.nvfp4moe_set_gemm_kernel(N.GEMM_AUTO)


# expert sizes cover: one full pair block, half-empty pair blocks (P_e / 128
# odd), empty experts, a single row, and widths that are not multiples of 256
@pytest.mark.parametrize("sizes,N_,K", [([256], 1024, 512), ([5, 0, 295, 130], 256, 512), ([1], 256, 256),
                                        ([200, 77], 384, 2048), ([128, 128, 0], 512, 1536),
                                        ([0, 700, 1, 0, 129], 768, 768)])
def test_nvfp4_fwd_within_bound(sizes, N_, K, gemm_kernel):
    y, xq, wq, o = _fwd(sizes, N_, K)
    A = _deq_nvfp4(xq, o)
    B = _deq_nvfp4(wq)
    if B.ndim == 2:
        B = B[None]
    y_ref, bound = G.grouped_rows(A, B, o)
    ok = G.within_bound(y.cpu().numpy(), y_ref, bound)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside the bound; max err {np.abs(y.cpu().numpy() - y_ref).max()}"


def test_nvfp4_fwd_bf16_output_and_determinism(gemm_kernel):
    y1, xq, wq, o = _fwd([5, 0, 295, 130], 256, 1024, out_fp32=False, seed=4)
    y2, _, _, _ = _fwd([5, 0, 295, 130], 256, 1024, out_fp32=False, seed=4)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    A, B = _deq_nvfp4(xq, o), _deq_nvfp4(wq)
    y_ref, bound = G.grouped_rows(A, B, o)
    assert G.within_bound(bf16_f32(y1), y_ref, bound, bf16_out=True).all()


def _mx_operands(sizes, Nd, K, seed):
    """g [M, Nd] (SR row-wise + transposed), w [E, Nd, K] -> NVFP4 -> requant
    transposed [E][K][Nd], x [M, K] -> NVFP4 -> requant transposed [K][P]."""
    go, o = _groups(sizes)
    M, E = int(o[-1]), len(sizes)
    g = _rand((M, Nd), seed, 1e-3)
    w = _rand((E, Nd, K), seed + 1, 0.02)
    x = _rand((M, K), seed + 2)
    wq, xq = NvTensor(E, Nd, K, dev()), NvTensor(1, M, K, dev(), E=E)
    wq.quantize(w)
    xq.quantize(x, go)
    wt, xt = MxTransposed(Nd, K, dev(), batch=E), MxTransposed(M, K, dev(), E=E)
    N.dequant_transpose_requant_sr(wq.codes, wq.scales, wq.sg, E, Nd, K, None, 3, 0, wt.codes, wt.scales)
    N.dequant_transpose_requant_sr(xq.codes, xq.scales, xq.sg, 1, M, K, go, 3, 2, xt.codes, xt.scales)
    gr, gt = MxRows(M, Nd, dev(), E=E), MxTransposed(M, Nd, dev(), E=E)
    N.mxfp8_quantize(g, M, Nd, go, N.NV_SR, 3, 4, 5, gr.codes, gr.scales, gt.codes, gt.scales)
    check_status()
    return go, o, M, E, gr, gt, wt, xt


# the last two cases have 200 wgrad pair tiles (10 experts x 4 x 5) and 256
# (one expert, 16 x 16): more than two rounds of the 76 CTA pairs, so the
# pair kernel's snake order walks a round in reverse and ends on a partial
# one, over experts of very different sizes and within a single expert
@pytest.mark.parametrize("sizes,Nd,K", [([256], 1024, 512), ([5, 0, 295, 130], 256, 384), ([1, 300], 128, 256),
                                       ([5, 0, 295, 130], 256, 512), ([0, 700, 1, 0, 129], 512, 768),
                                       ([300, 0, 5, 129, 700, 1, 256, 0, 33, 128], 1024, 1280),
                                       ([200], 4096, 4096)])
def test_mxfp8_dgrad_and_wgrad_within_bound(sizes, Nd, K, gemm_kernel):
    go, o, M, E, gr, gt, wt, xt = _mx_operands(sizes, Nd, K, seed=len(sizes) + Nd)
    dx = gfull((M, K), float("nan"), dtype=torch.float32, device=dev())
    dw = gfull((E, Nd, K), float("nan"), dtype=torch.float32, device=dev())
    N.grouped_gemm_mxfp8_dx(gr.codes, gr.scales, wt.codes, wt.scales, go, E, M, Nd, K, dx, N.NV_OUT_FP32)
    N.grouped_gemm_mxfp8_dw(gt.codes, gt.scales, xt.codes, xt.scales, go, E, M, Nd, K, dw)
    check_status()
    # dgrad: A = g rows (grouped scales), B_e = w_e^T [K, Nd]
    g64 = MX.dequantize_f64(gr.codes[: M * Nd].cpu().numpy().reshape(M, Nd),
                            L.unswizzle(gr.scales.cpu().numpy(), L.grouped_row_map(o), Nd // 32))
    wt64 = MX.dequantize_f64(wt.codes[: E * K * Nd].cpu().numpy().reshape(E * K, Nd),
                             L.unswizzle(wt.scales.cpu().numpy(), L.batched_row_map(E, K), Nd // 32)).reshape(E, K, Nd)
    dx_ref, dx_bound = G.grouped_rows(g64, wt64, o)
    okx = G.within_bound(dx.cpu().numpy(), dx_ref, dx_bound)
    assert okx.all(), f"dgrad: {(~okx).sum()} outside"
    # wgrad: A = g^T [Nd, P], B = x_q^T [K, P]
    P = gt.P
    gt64 = MX.dequantize_f64(gt.codes[: Nd * P].cpu().numpy().reshape(Nd, P),
                             L.unswizzle(gt.scales.cpu().numpy(), np.arange(Nd), P // 32))
    xt64 = MX.dequantize_f64(xt.codes[: K * P].cpu().numpy().reshape(K, P),
                             L.unswizzle(xt.scales.cpu().numpy(), np.arange(K), P // 32))
    Ps = L.group_padded_starts(o)
    dw_ref, dw_bound = G.grouped_contraction(gt64, xt64, Ps)
    okw = G.within_bound(dw.cpu().numpy(), dw_ref, dw_bound)
    assert okw.all(), f"wgrad: {(~okw).sum()} outside"
    empty = [e for e, s in enumerate(sizes) if s == 0]
    for e in empty:
        assert torch.all(dw[e] == 0)


def test_single_linear_layer_end_to_end():
    s = W.single_linear("cuda")
    layer = SingleLinear(256, 512, 1024)
    out = layer.run(s.x, s.w, s.g, seed=0)
    check_status()
    out2 = layer.run(s.x, s.w, s.g, seed=0)
    for k in ("y", "dx", "dw", "wt_codes", "gt_codes", "xt_codes"):
        assert np.array_equal(out[k], out2[k]), k
    xq, wq = layer.xq, layer.wq
    A, B = _deq_nvfp4(xq, np.array([0, 256])), _deq_nvfp4(wq)
    y_ref, bound = G.grouped_rows(A, B[None] if B.ndim == 2 else B, np.array([0, 256]))
    assert G.within_bound(out["y"], y_ref, bound).all()


@pytest.mark.parametrize("given_scale", [False, True])
def test_fwd_from_bf16_activations_equals_quantize_then_gemm(given_scale):
    """grouped_gemm_nvfp4_fwd given bf16 activations quantizes them itself
    (into its workspace) with nvfp4_quantize's rule: the output equals the
    two calls in sequence, bit for bit."""
    from precision_moe_numerics_nvfp4_gb300.pipeline import NvTensor
    sizes, N_, K = [37, 0, 200, 129], 256, 512
    o = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    go = torch.from_numpy(o).cuda()
    M, E = int(o[-1]), len(sizes)
    g = torch.Generator(device="cuda").manual_seed(41)
    x = torch.randn((M, K), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((E, N_, K), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    wq = NvTensor(E, N_, K, torch.device("cuda"))
    wq.quantize(w)
    sg_in = torch.tensor([0.75], dtype=torch.float32, device="cuda") if given_scale else None
    xq = NvTensor(1, M, K, torch.device("cuda"), E=E)
    xq.quantize(x, go, sg_in=sg_in)
    y_ref = gempty((M, N_), dtype=torch.float32, device="cuda")
    N.grouped_gemm_nvfp4_fwd(None, xq.sg, xq.codes, xq.scales, wq.codes, wq.scales, wq.sg, go, E, M, N_, K, y_ref,
                             N.NV_OUT_FP32)
    ws = gempty(N.nvfp4moe_fwd_workspace_bytes(M, K, E), dtype=torch.uint8, device="cuda")
    y = gfull((M, N_), 7.0, dtype=torch.float32, device="cuda")
    N.grouped_gemm_nvfp4_fwd(x, sg_in, None, None, wq.codes, wq.scales, wq.sg, go, E, M, N_, K, y, N.NV_OUT_FP32,
                             workspace=ws)
    assert N.nvfp4moe_get_device_status() == 0
    assert torch.equal(y, y_ref)
