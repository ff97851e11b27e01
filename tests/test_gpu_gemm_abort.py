"""The grouped GEMMs' bounded-wait path on the GPU (the one-CTA kernel, in
which one thread issues every copy of the CTA and waits for them).  With the
pipeline waits limited to a single poll, waits run out: the kernel must
record NV_ERR_TIMEOUT in the status word and leave on its own (the copies and
MMAs it has in flight are waited for with their own bound before tensor
memory is freed), with no fault and no hang; afterwards the same GEMM with
the default limit must again give the full, correct result, so the context
is still usable.  NVFP4 forward, MXFP8 dgrad and MXFP8 wgrad."""
import numpy as np
import pytest
import torch

from oracle import gemm as G
from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
from tests.test_gpu_gemm import _deq_nvfp4, _fwd, _mx_operands
from tests.gpu_helpers import check_status, dev, gfull

pytestmark = pytest.mark.gpu

SIZES, N_, K = [256, 300, 0, 512], 512, 1024


@pytest.fixture
def one_cta_kernel():
    N.nvfp4moe_set_gemm_kernel(N.GEMM_TWO_PER_SM)
    yield
    N.nvfp4moe_set_gemm_wait_limit(0)
    N.nvfp4moe_set_gemm_kernel(N.GEMM_AUTO)


def _statuses_with_one_poll(launch, attempts=6):
    out = []
    N.nvfp4moe_set_gemm_wait_limit(1)
    try:
        for _ in range(attempts):
            launch()
            torch.cuda.synchronize()
            out.append(N.nvfp4moe_get_device_status())
    finally:
        N.nvfp4moe_set_gemm_wait_limit(0)
    return out


def test_nvfp4_fwd_wait_runs_out_then_recovers(one_cta_kernel):
    y, xq, wq, o = _fwd(SIZES, N_, K)  # operands (and a first, healthy run)
    go = torch.from_numpy(o.astype(np.int32)).to(dev())
    M, E = int(o[-1]), len(SIZES)
    y2 = gfull((M, N_), float("nan"), dtype=torch.float32, device=dev())
    launch = lambda: N.grouped_gemm_nvfp4_fwd(None, xq.sg, xq.codes, xq.scales, wq.codes, wq.scales, wq.sg, go, E, M,
                                              N_, K, y2, N.NV_OUT_FP32)
    st = _statuses_with_one_poll(launch)
    assert all(s in (N.NV_OK, N.NV_ERR_TIMEOUT) for s in st), st
    assert N.NV_ERR_TIMEOUT in st, st
    # the context is usable: the default limit gives the full, correct result
    launch()
    check_status()
    y_ref, bound = G.grouped_rows(_deq_nvfp4(xq, o), _deq_nvfp4(wq), o)
    assert G.within_bound(y2.cpu().numpy(), y_ref, bound).all()
    assert torch.equal(y2, y)


@pytest.mark.parametrize("which", ["dgrad", "wgrad"])
def test_mxfp8_wait_runs_out_then_recovers(which, one_cta_kernel):
    Nd = 512
    go, o, M, E, gr, gt, wt, xt = _mx_operands(SIZES, Nd, K, seed=11)
    if which == "dgrad":
        out = gfull((M, K), float("nan"), dtype=torch.float32, device=dev())
        launch = lambda: N.grouped_gemm_mxfp8_dx(gr.codes, gr.scales, wt.codes, wt.scales, go, E, M, Nd, K, out,
                                                 N.NV_OUT_FP32)
    else:
        out = gfull((E, Nd, K), float("nan"), dtype=torch.float32, device=dev())
        launch = lambda: N.grouped_gemm_mxfp8_dw(gt.codes, gt.scales, xt.codes, xt.scales, go, E, M, Nd, K, out)
    launch()  # a healthy run first: the reference result
    check_status()
    ref = out.clone()
    assert not torch.isnan(ref).any()
    st = _statuses_with_one_poll(launch)
    assert all(s in (N.NV_OK, N.NV_ERR_TIMEOUT) for s in st), st
    assert N.NV_ERR_TIMEOUT in st, st
    out.fill_(float("nan"))
    launch()  # the default limit again: the same bits as the healthy run
    check_status()
    assert torch.equal(out, ref)
