"""nvfp4_quantize_noalloc: the variant of nvfp4_quantize for callers that
cannot allocate device memory (it uses the library's fixed scratch instead of
a workspace).  Its output must equal the workspace entry point's, bit for bit,
on two calls in a row; requests beyond the scratch are refused on the host.
This file sorts last so that a run stopping at the first failure has already
run everything else; it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N

pytestmark = pytest.mark.gpu


def _input(shape, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * 0.05).to(torch.bfloat16).contiguous()


def _run(fn_name, x, batch, rows, cols, groups=None, sg_in=None, want_sg=True):
    """Codes, scales and (when want_sg) the outer scales the call wrote."""
    E = None if groups is None else groups.numel() - 1
    cb, sb = N.nvfp4_sizes(batch, rows, cols, E)
    codes = torch.full((cb,), 0xA5, dtype=torch.uint8, device="cuda")
    scales = torch.full((sb,), 0xA5, dtype=torch.uint8, device="cuda")
    sg = torch.full((batch,), -1.0, dtype=torch.float32, device="cuda") if want_sg else None
    if fn_name == "nvfp4_quantize":
        ws = torch.zeros(N.nvfp4moe_quantize_workspace_bytes(batch, rows, cols), dtype=torch.uint8, device="cuda")
        N.nvfp4_quantize(x, batch, rows, cols, groups, sg_in, sg, codes, scales, None if sg_in is not None else ws)
    else:
        N.nvfp4_quantize_noalloc(x, batch, rows, cols, groups, sg_in, sg, codes, scales)
    assert N.nvfp4moe_get_device_status() == 0
    out = [codes.cpu().numpy(), scales.cpu().numpy()]
    if want_sg:
        out.append(sg.cpu().numpy())
    return out


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    groups = torch.tensor([0, 5, 5, 300, 428], dtype=torch.int32, device="cuda")
    cases = [(_input((3, 200, 160), 1), 3, 200, 160, None),      # batched, three outer scales
             (_input((428, 256), 2), 1, 428, 256, groups)]        # grouped rows, smaller
    for x, batch, rows, cols, go in cases:                         # two calls in a row
        ref = _run("nvfp4_quantize", x, batch, rows, cols, go)
        got = _run("nvfp4_quantize_noalloc", x, batch, rows, cols, go)
        for a, b in zip(ref, got):
            assert np.array_equal(a, b)


def test_noalloc_without_outer_scale_output():
    # outer_scale_out NULL: the outer scales then live in the shared scratch
    # itself, between the amax pass and the quantizer that reads them
    x = _input((2, 256, 192), 3)
    for _ in range(2):
        ref = _run("nvfp4_quantize", x, 2, 256, 192, want_sg=False)
        got = _run("nvfp4_quantize_noalloc", x, 2, 256, 192, want_sg=False)
        for a, b in zip(ref, got):
            assert np.array_equal(a, b)


def test_noalloc_with_given_outer_scale_has_no_size_limit():
    # outer_scale_in set: no amax pass, no scratch, so a shape whose workspace
    # would exceed the scratch (26216 matrices of 128 x 512, 3.4 GB of bf16)
    # is accepted and matches the workspace entry point; compared on the device
    batch, rows, cols = 26216, 128, 512
    assert N.nvfp4moe_quantize_workspace_bytes(batch, rows, cols) > 524288
    x = _input((batch, rows, cols), 4)
    sg_in = torch.linspace(0.5, 2.0, batch, device="cuda", dtype=torch.float32)
    cb, sb = N.nvfp4_sizes(batch, rows, cols, None)
    outs = []
    for fn in ("nvfp4_quantize", "nvfp4_quantize_noalloc"):
        codes = torch.full((cb,), 0xA5, dtype=torch.uint8, device="cuda")
        scales = torch.full((sb,), 0xA5, dtype=torch.uint8, device="cuda")
        sg = torch.full((batch,), -1.0, dtype=torch.float32, device="cuda")
        if fn == "nvfp4_quantize":
            N.nvfp4_quantize(x, batch, rows, cols, None, sg_in, sg, codes, scales, None)
        else:
            N.nvfp4_quantize_noalloc(x, batch, rows, cols, None, sg_in, sg, codes, scales)
        assert N.nvfp4moe_get_device_status() == 0
        outs.append((codes, scales, sg))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    assert torch.equal(outs[1][2], sg_in)
    assert not torch.all(outs[1][0] == 0xA5)   # the codes were written


def test_noalloc_refuses_requests_beyond_its_scratch():
    # 1024 matrices of 16384 x 256: needs more partial maxima than the scratch holds
    batch, rows, cols = 1024, 16384, 256
    assert N.nvfp4moe_quantize_workspace_bytes(batch, rows, cols) > 524288
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")  # never read: refused before any launch
    buf = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(N.NvError) as e:
        N.nvfp4_quantize_noalloc(x, batch, rows, cols, None, None, None, buf, buf)
    assert e.value.status == N.NV_ERR_WORKSPACE
