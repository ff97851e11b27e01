"""grouped_gemm_nvfp4_fwd_swiglu against the unfused sequence, bit for bit:
y13 = grouped_gemm_nvfp4_fwd (bf16 output), h = nvfp4moe_swiglu_fwd(y13), and
h's outer scale = the one nvfp4_quantize computes for h; ragged and empty
groups, several hidden sizes; and a whole MoE step with and without the fused
epilogue gives identical outputs."""
import numpy as np
import pytest
import torch

from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
from precision_moe_numerics_nvfp4_gb300 import pipeline as PL
from precision_moe_numerics_nvfp4_gb300 import workloads as W
from precision_moe_numerics_nvfp4_gb300.pipeline import NvTensor
from tests.gpu_helpers import check_status, dev, gempty, gfull

pytestmark = pytest.mark.gpu


def _rand(shape, seed, std):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * std).to(torch.bfloat16).contiguous()


@pytest.fixture(params=[N.GEMM_AUTO, N.GEMM_TWO_PER_SM, N.GEMM_CTA_PAIR], ids=["auto", "two_per_sm", "cta_pair"])
def gemm_kernel(request):
    """The fused epilogue exists in the 128 x 128 kernel and in the CTA-pair
    kernel (128 gate + 128 up rows per pair tile); both must match the
    unfused sequence run with the same kernel choice."""
    N.nvfp4moe_set_gemm_kernel(request.param)
    yield request.param
    N.nvfp4moe_set_gemm_kernel(N.GEMM_AUTO)


@pytest.mark.parametrize("sizes,I,K", [([300], 128, 256), ([5, 0, 295, 130, 1], 256, 512), ([0, 700, 0], 384, 256),
                                       ([128, 128], 1536, 1024), ([600, 1, 0, 257, 513], 256, 512)])
def test_fused_swiglu_equals_unfused(sizes, I, K, gemm_kernel):
    o = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    go = torch.from_numpy(o).to(dev())
    M, E = int(o[-1]), len(sizes)
    x = _rand((M, K), 1 + I, 1.0)
    w13 = _rand((E, 2 * I, K), 2 + I, 0.05)
    xq, wq = NvTensor(1, M, K, dev(), E=E), NvTensor(E, 2 * I, K, dev())
    xq.quantize(x, go)
    wq.quantize(w13)
    y_ref = gfull((M, 2 * I), 7, dtype=torch.bfloat16, device=dev())
    h_ref = gfull((M, I), 7, dtype=torch.bfloat16, device=dev())
    N.grouped_gemm_nvfp4_fwd(None, xq.sg, xq.codes, xq.scales, wq.codes, wq.scales, wq.sg, go, E, M, 2 * I, K, y_ref,
                             N.NV_OUT_BF16)
    N.nvfp4moe_swiglu_fwd(y_ref, M, I, h_ref)
    hq = NvTensor(1, M, I, dev(), E=E)
    hq.quantize(h_ref, go)
    y = gfull((M, 2 * I), 9, dtype=torch.bfloat16, device=dev())
    h = gfull((M, I), 9, dtype=torch.bfloat16, device=dev())
    sg = gfull((1,), -1.0, dtype=torch.float32, device=dev())
    N.grouped_gemm_nvfp4_fwd_swiglu(xq.sg, xq.codes, xq.scales, wq.codes, wq.scales, wq.sg, go, E, M, I, K, y, h, sg)
    check_status()
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    assert torch.equal(h.view(torch.int16), h_ref.view(torch.int16))
    assert torch.equal(sg, hq.sg)


def test_fused_swiglu_rejects_bad_shapes():
    go = torch.tensor([0, 128], dtype=torch.int32, device=dev())
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device=dev())
    sg = torch.ones(1, dtype=torch.float32, device=dev())
    with pytest.raises(N.NvError):  # I % 128 != 0
        N.grouped_gemm_nvfp4_fwd_swiglu(sg, buf, buf, buf, buf, sg, go, 1, 128, 64, 256, buf, buf, sg)
    with pytest.raises(N.NvError):  # 16-byte but not 32-byte aligned output
        N.grouped_gemm_nvfp4_fwd_swiglu(sg, buf, buf, buf, buf, sg, go, 1, 128, 128, 256, buf[16:], buf, sg)


def test_moe_step_same_with_and_without_fused_epilogue():
    d, I, E, tokens = 512, 256, 8, 512
    m = W.moe("cuda", seed=7, tokens=tokens, d_model=d, experts=E, topk=2, d_ff=I, with_grad=True, grad_seed=8)
    M = m.x_perm.shape[0]
    outs = []
    for fuse in (True, False):
        layer = PL.MoELayer(M, d, I, E, fuse_swiglu=fuse)
        assert layer.fuse_swiglu == fuse
        layer.step(m.x_perm, m.w13, m.w2, m.g2, m.group_offsets, seed=3)
        torch.cuda.synchronize()
        outs.append({k: getattr(layer, k).clone() for k in ("y13", "h", "y2", "dx", "dw13", "dw2")})
        outs[-1]["hq"] = layer.hq.codes.clone()
        # the transposed h: columns past the experts' padded tokens are left
        # untouched by the library (their bytes are whatever the buffer held)
        sizes = torch.diff(m.group_offsets.to(torch.int64)).cpu()
        P_total = int(((sizes + 127) // 128 * 128).sum())
        P_cap = layer.ht.P
        outs[-1]["ht"] = layer.ht.codes[: I * P_cap].view(I, P_cap)[:, :P_total].clone()
    check_status()
    for k in outs[0]:
        a, b = outs[0][k], outs[1][k]
        assert torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                           b.view(torch.uint8) if b.dtype != torch.uint8 else b), k
