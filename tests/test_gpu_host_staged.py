"""HostStaged runs MoE layer steps from pinned host buffers with the copies of
neighbouring steps overlapping the compute; its dx must be bit-identical to
the same steps run on device-resident inputs, step by step, while slots and
streams are reused (more steps than slots, different inputs per step)."""
import pytest
import torch

from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
from precision_moe_numerics_nvfp4_gb300 import pipeline as PL
from precision_moe_numerics_nvfp4_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_host_staged_matches_device_steps():
    d, I, E, tokens = 512, 256, 8, 512
    base = W.moe("cuda", seed=5, tokens=tokens, d_model=d, experts=E, topk=2, d_ff=I, with_grad=True, grad_seed=6)
    M = base.x_perm.shape[0]
    gen = torch.Generator(device="cuda").manual_seed(11)
    xs = [(torch.randn((M, d), generator=gen, device="cuda")).to(torch.bfloat16) for _ in range(5)]
    gs = [(torch.randn((M, d), generator=gen, device="cuda") * 1e-3).to(torch.bfloat16) for _ in range(5)]
    ref_layer = PL.MoELayer(M, d, I, E)
    want = []
    for x, g in zip(xs, gs):
        ref_layer.step(x, base.w13, base.w2, g, base.group_offsets, seed=3)
        want.append(ref_layer.dx.clone())
    torch.cuda.synchronize()

    layer = PL.MoELayer(M, d, I, E)
    staged = PL.HostStaged(layer)
    x_h = [x.cpu().pin_memory() for x in xs]
    g_h = [g.cpu().pin_memory() for g in gs]
    dx_h = [torch.empty((M, d), dtype=torch.bfloat16).pin_memory() for _ in xs]
    for k in range(len(xs)):
        staged.step(x_h[k], g_h[k], dx_h[k], base.w13, base.w2, base.group_offsets, seed=3)
    staged.synchronize()
    torch.cuda.synchronize()
    assert N.nvfp4moe_get_device_status() == 0
    for k in range(len(xs)):
        assert torch.equal(dx_h[k].view(torch.int16), want[k].cpu().view(torch.int16)), f"step {k}"
    assert staged.bytes_per_step() == (2 * M * d * 2, M * d * 2)


def test_host_staged_from_tokens_matches_device_steps():
    """The same with the tokens and the routed rows' source map as inputs
    (the quantization of x gathers the routed rows)."""
    d, I, E, tokens = 512, 256, 8, 512
    base = W.moe("cuda", seed=5, tokens=tokens, d_model=d, experts=E, topk=2, d_ff=I, with_grad=True, grad_seed=6)
    M = base.x_perm.shape[0]
    gen = torch.Generator(device="cuda").manual_seed(12)
    xs = [(torch.randn((tokens, d), generator=gen, device="cuda")).to(torch.bfloat16) for _ in range(4)]
    rs = [torch.randint(0, tokens, (M,), generator=gen, device="cuda", dtype=torch.int32) for _ in range(4)]
    gs = [(torch.randn((M, d), generator=gen, device="cuda") * 1e-3).to(torch.bfloat16) for _ in range(4)]
    ref_layer = PL.MoELayer(M, d, I, E)
    want = []
    for x, r, g in zip(xs, rs, gs):
        ref_layer.step(x[r.long()].contiguous(), base.w13, base.w2, g, base.group_offsets, seed=3)
        want.append(ref_layer.dx.clone())
    torch.cuda.synchronize()
    layer = PL.MoELayer(M, d, I, E)
    staged = PL.HostStaged(layer, tokens=tokens)
    x_h = [x.cpu().pin_memory() for x in xs]
    r_h = [r.cpu().pin_memory() for r in rs]
    g_h = [g.cpu().pin_memory() for g in gs]
    dx_h = [torch.empty((M, d), dtype=torch.bfloat16).pin_memory() for _ in xs]
    for k in range(len(xs)):
        staged.step(x_h[k], g_h[k], dx_h[k], base.w13, base.w2, base.group_offsets, seed=3, rows_h=r_h[k])
    staged.synchronize()
    torch.cuda.synchronize()
    assert N.nvfp4moe_get_device_status() == 0
    for k in range(len(xs)):
        assert torch.equal(dx_h[k].view(torch.int16), want[k].cpu().view(torch.int16)), f"step {k}"
    assert staged.bytes_per_step() == (tokens * d * 2 + M * 4 + M * d * 2, M * d * 2)
