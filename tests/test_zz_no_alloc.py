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


def _run(fn_name, x, batch, rows, cols, groups=None):
    E = None if groups is None else groups.numel() - 1
    cb, sb = N.nvfp4_sizes(batch, rows, cols, E)
    codes = torch.full((cb,), 0xA5, dtype=torch.uint8, device="cuda")
    scales = torch.full((sb,), 0xA5, dtype=torch.uint8, device="cuda")
    sg = torch.full((batch,), -1.0, dtype=torch.float32, device="cuda")
    if fn_name == "nvfp4_quantize":
        ws = torch.zeros(N.nvfp4moe_quantize_workspace_bytes(batch, rows, cols), dtype=torch.uint8, device="cuda")
        N.nvfp4_quantize(x, batch, rows, cols, groups, None, sg, codes, scales, ws)
    else:
        N.nvfp4_quantize_noalloc(x, batch, rows, cols, groups, None, sg, codes, scales)
    assert N.nvfp4moe_get_device_status() == 0
    return codes.cpu().numpy(), scales.cpu().numpy(), sg.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    groups = torch.tensor([0, 5, 5, 300, 428], dtype=torch.int32, device="cuda")
    cases = [(_input((3, 200, 160), 1), 3, 200, 160, None),      # batched, three outer scales
             (_input((428, 256), 2), 1, 428, 256, groups)]        # grouped rows, smaller
    for x, batch, rows, cols, go in cases:                         # two calls in a row
        ref = _run("nvfp4_quantize", x, batch, rows, cols, go)
        got = _run("nvfp4_quantize_noalloc", x, batch, rows, cols, go)
        for a, b in zip(ref, got):
            assert np.array_equal(a, b)


def test_noalloc_refuses_requests_beyond_its_scratch():
    # 1024 matrices of 16384 x 256: needs more partial maxima than the scratch holds
    batch, rows, cols = 1024, 16384, 256
    assert N.nvfp4moe_quantize_workspace_bytes(batch, rows, cols) > 524288
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")  # never read: refused before any launch
    buf = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(N.NvError) as e:
        N.nvfp4_quantize_noalloc(x, batch, rows, cols, None, None, None, buf, buf)
    assert e.value.status == N.NV_ERR_WORKSPACE
