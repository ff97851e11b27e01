"""nvfp4_quantize_requant_gather (the expert dispatch folded into the
quantization of x): quantizing the routed-row matrix X[r] = x[row_src[r]]
without materializing it must give exactly what nvfp4_quantize_requant gives
on the materialized X (codes, scales, outer scale, MXFP8 codes and scales),
with the outer scale computed or given, for ragged and empty expert groups;
an index outside the token range reads as zeros and is recorded; and a MoE
layer step fed the tokens and the routing equals the step fed the routed
rows, bit for bit."""
import numpy as np
import pytest
import torch

from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
from precision_moe_numerics_nvfp4_gb300 import pipeline as PL
from precision_moe_numerics_nvfp4_gb300 import workloads as W
from precision_moe_numerics_nvfp4_gb300.pipeline import MxTransposed, NvTensor
from tests.gpu_helpers import check_status, dev

pytestmark = pytest.mark.gpu


def _pair(M, K, E):
    a, b = NvTensor(1, M, K, dev(), E=E), NvTensor(1, M, K, dev(), E=E)
    ma, mb = MxTransposed(M, K, dev(), E=E), MxTransposed(M, K, dev(), E=E)
    for t in (a.codes, a.scales, b.codes, b.scales, ma.codes, ma.scales, mb.codes, mb.scales):
        t.fill_(0xA5)
    return a, b, ma, mb


# the amax pass: tokens read once (T <= M) or the routed rows read (T > M)
@pytest.mark.parametrize("sizes,T,K,given", [([5, 0, 295, 130], 300, 256, False), ([128, 1, 0, 257], 97, 512, True),
                                             ([0, 640], 640, 128, False), ([40, 0, 24], 1000, 256, False),
                                             ([128, 1, 0, 257], 97, 512, False), ([40, 0, 24], 1000, 256, True)])
def test_gather_equals_materialized_rows(sizes, T, K, given):
    g = torch.Generator(device="cuda").manual_seed(sum(sizes) + K)
    x = (torch.randn((T, K), generator=g, device="cuda") * 3).to(torch.bfloat16)
    x[0, 5] = 3.0e4  # token 0 is routed nowhere: its maximum must not reach the outer scale
    M = int(sum(sizes))
    rows = torch.randint(1, T, (M,), generator=g, device="cuda", dtype=torch.int32)
    groups = torch.tensor(np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32), device=dev())
    E = len(sizes)
    xp = x[rows.long()].contiguous()
    a, b, ma, mb = _pair(M, K, E)
    sg_in = torch.tensor([0.125], dtype=torch.float32, device=dev()) if given else None
    N.nvfp4_quantize_requant(xp, 1, M, K, groups, sg_in, a.sg, a.codes, a.scales, a.ws, 3, 2, ma.codes, ma.scales)
    N.nvfp4_quantize_requant_gather(x, rows, T, M, K, groups, sg_in, b.sg, b.codes, b.scales,
                                    b.gather_workspace(T), 3, 2, mb.codes, mb.scales)
    check_status()
    for u, v in ((a.sg, b.sg), (a.codes, b.codes), (a.scales, b.scales), (ma.codes, mb.codes),
                 (ma.scales, mb.scales)):
        assert torch.equal(u, v)


@pytest.mark.parametrize("T", [64, 100])
def test_gather_index_out_of_range_reads_zeros_and_is_recorded(T):
    K, sizes = 128, [40, 24]
    g = torch.Generator(device="cuda").manual_seed(5)
    x = torch.randn((T, K), generator=g, device="cuda").to(torch.bfloat16)
    M = sum(sizes)
    rows = torch.randint(0, T, (M,), generator=g, device="cuda", dtype=torch.int32)
    rows[7] = T          # one past the end
    rows[50] = -3
    groups = torch.tensor([0, 40, 64], dtype=torch.int32, device=dev())
    xp = x[rows.clamp(0, T - 1).long()].clone()
    xp[7] = 0
    xp[50] = 0
    a, b, ma, mb = _pair(M, K, 2)
    N.nvfp4_quantize_requant(xp, 1, M, K, groups, None, a.sg, a.codes, a.scales, a.ws, 3, 2, ma.codes, ma.scales)
    check_status()
    N.nvfp4_quantize_requant_gather(x, rows, T, M, K, groups, None, b.sg, b.codes, b.scales,
                                    b.gather_workspace(T), 3, 2, mb.codes, mb.scales)
    assert N.nvfp4moe_get_device_status() == N.NV_ERR_ARG
    for u, v in ((a.sg, b.sg), (a.codes, b.codes), (a.scales, b.scales), (ma.codes, mb.codes)):
        assert torch.equal(u, v)


def test_layer_step_from_tokens_equals_step_from_routed_rows():
    d, I, E, tokens = 512, 256, 8, 512
    m = W.moe("cuda", seed=9, tokens=tokens, d_model=d, experts=E, topk=2, d_ff=I, with_grad=True, grad_seed=10)
    M = m.x_perm.shape[0]
    outs = []
    for gather in (False, True):
        layer = PL.MoELayer(M, d, I, E)
        if gather:
            layer.step(m.x, m.w13, m.w2, m.g2, m.group_offsets, seed=3, x_rows=m.rows)
        else:
            layer.step(m.x_perm, m.w13, m.w2, m.g2, m.group_offsets, seed=3)
        torch.cuda.synchronize()
        outs.append([t.clone() for t in (layer.xq.codes, layer.xq.scales, layer.xq.sg, layer.y2, layer.dx,
                                          layer.dw13, layer.dw2)])
    check_status()
    for u, v in zip(*outs):
        assert torch.equal(u.view(torch.uint8), v.view(torch.uint8))


@pytest.mark.parametrize("sizes,T,K", [([5, 0, 295, 130], 300, 256), ([40, 0, 24], 1000, 128)])
def test_gather_against_the_oracle(sizes, T, K):
    """The gathered call held directly to the oracle quantizing X = x[row_src]:
    NVFP4 codes, block scales and outer scale exact, and the transposed SR
    re-quantization exact (draws keyed by the routed row), for both amax
    paths (T <= M reads each token once, T > M the routed rows)."""
    from oracle import layout as L
    from oracle import nvfp4 as NV
    from oracle import requant as RQ
    from tests.gpu_helpers import oracle_nvfp4, unpack_gpu_nvfp4
    g = torch.Generator(device="cuda").manual_seed(T + K)
    x = (torch.randn((T, K), generator=g, device="cuda") * 2).to(torch.bfloat16)
    M = int(sum(sizes))
    rows = torch.randint(0, T, (M,), generator=g, device="cuda", dtype=torch.int32)
    o = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    groups = torch.tensor(o, device=dev())
    E = len(sizes)
    q, mt = NvTensor(1, M, K, dev(), E=E), MxTransposed(M, K, dev(), E=E)
    N.nvfp4_quantize_requant_gather(x, rows, T, M, K, groups, None, q.sg, q.codes, q.scales,
                                    q.gather_workspace(T), 7, 2, mt.codes, mt.scales)
    check_status()
    X = x.float().cpu().numpy()[rows.long().cpu().numpy()]  # the routed rows, gathered on the host
    codes, scales, sg = oracle_nvfp4(X, 1, M, K, groups=o)
    assert np.array_equal(q.sg.cpu().numpy(), sg)
    assert np.array_equal(q.codes.cpu().numpy()[: codes.size], codes)
    got_c, got_s = unpack_gpu_nvfp4(q.codes.cpu().numpy(), q.scales.cpu().numpy(), 1, M, K, o)
    want_c, want_s, _ = NV.quantize(X, sg[0])
    assert np.array_equal(got_c, want_c) and np.array_equal(got_s, want_s)
    P = N.nvfp4moe_padded_cap(M, E)
    ec, es = RQ.requant_grouped(want_c, want_s, sg[0], o, 7, 2, P)
    Ptot = int(L.group_padded_starts(o)[-1])
    assert np.array_equal(mt.codes.cpu().numpy()[: K * P].reshape(K, P)[:, :Ptot], ec[:, :Ptot])
    assert np.array_equal(L.unswizzle(mt.scales.cpu().numpy(), np.arange(K), P // 32), es)
