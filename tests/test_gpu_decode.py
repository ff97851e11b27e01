"""Full-size parity of the sampler-style decode forward: 128 experts with
SwiGLU gate/up [7168 -> 2048 x2] and down [2048 -> 7168], NVFP4 weights
quantized beforehand, 256 tokens routed top-8 (1..64 rows per expert).  The
forward (NVFP4 quantization of x, grouped NVFP4 GEMM w13, SwiGLU, quantization
of h, grouped NVFP4 GEMM w2) runs as bench.py times it; sampled rows of every
stage are compared with the oracle fed the GPU's own stage input."""
import numpy as np
import pytest
import torch

from oracle import gemm as G
from oracle import layout as L
from oracle import nvfp4 as NV
from oracle import swiglu as SW
from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
from precision_moe_numerics_nvfp4_gb300 import pipeline as PL
from precision_moe_numerics_nvfp4_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_decode_forward_full_size():
    m = W.decode("cuda")
    M, D, I, E = m.x_perm.shape[0], 7168, 2048, 128
    layer = PL.MoELayer(M, D, I, E, backward=False)
    layer.quantize_weights(m.w13, m.w2)
    layer.forward_activations(m.x_perm, m.group_offsets)
    torch.cuda.synchronize()
    assert N.nvfp4moe_get_device_status() == 0
    o = m.group_offsets.cpu().numpy().astype(np.int64)
    sizes = np.diff(o)
    assert sizes.min() >= 1 and sizes.max() <= 64
    rmap = L.grouped_row_map(o)
    rng = np.random.default_rng(5)
    experts = [int(np.argmax(sizes)), int(np.argmin(sizes))] + [int(e) for e in rng.choice(E, 2, replace=False)]
    sgx, sgh = layer.xq.sg.cpu().numpy()[0], layer.hq.sg.cpu().numpy()[0]
    xf = m.x_perm.float().cpu().numpy()
    assert sgx == NV.outer_scale(xf)
    h_all = layer.h.float().cpu().numpy()
    assert sgh == NV.outer_scale(h_all)
    for e in experts:
        rows = np.arange(o[e], o[e + 1])
        # x_q of the expert's rows, bit-exact
        codes = layer.xq.codes[: M * D // 2].view(M, D // 2)[torch.as_tensor(rows, device="cuda")]
        xc = NV.unpack(codes.cpu().numpy())
        xs = L.unswizzle(layer.xq.scales.cpu().numpy(), rmap[rows], D // 16)
        ec, es, _ = NV.quantize(xf[rows], sgx)
        assert np.array_equal(xc, ec) and np.array_equal(xs, es)
        # weights of the expert, bit-exact, and the two GEMMs within the bound
        wc = NV.unpack(layer.w13q.codes[: E * 2 * I * D // 2].view(E, 2 * I, D // 2)[e].cpu().numpy())
        ws = L.unswizzle(layer.w13q.scales.cpu().numpy(), e * 2 * I + np.arange(2 * I), D // 16)
        wsg = layer.w13q.sg.cpu().numpy()[e]
        if e == experts[0]:
            ewc, ews, ewsg = NV.quantize(m.w13[e].float().cpu().numpy())
            assert wsg == ewsg and np.array_equal(wc, ewc) and np.array_equal(ws, ews)
        y_ref, bound = G.grouped_rows(NV.dequantize_f64(xc, xs, sgx), NV.dequantize_f64(wc, ws, wsg)[None],
                                      np.array([0, len(rows)]))
        y13 = layer.y13[torch.as_tensor(rows, device="cuda")].float().cpu().numpy()
        assert G.within_bound(y13, y_ref, bound, bf16_out=True).all()
        h = h_all[rows]
        h_ref = SW.forward(y13.astype(np.float64))
        assert np.all(np.abs(h - h_ref) <= np.abs(h_ref) * 2.0 ** -7 + 1e-30)
        hcodes = layer.hq.codes[: M * I // 2].view(M, I // 2)[torch.as_tensor(rows, device="cuda")]
        hc = NV.unpack(hcodes.cpu().numpy())
        hs = L.unswizzle(layer.hq.scales.cpu().numpy(), rmap[rows], I // 16)
        ec, es, _ = NV.quantize(h, sgh)
        assert np.array_equal(hc, ec) and np.array_equal(hs, es)
        w2c = NV.unpack(layer.w2q.codes[: E * D * I // 2].view(E, D, I // 2)[e].cpu().numpy())
        w2s = L.unswizzle(layer.w2q.scales.cpu().numpy(), e * D + np.arange(D), I // 16)
        y_ref, bound = G.grouped_rows(NV.dequantize_f64(hc, hs, sgh),
                                      NV.dequantize_f64(w2c, w2s, layer.w2q.sg.cpu().numpy()[e])[None],
                                      np.array([0, len(rows)]))
        y2 = layer.y2[torch.as_tensor(rows, device="cuda")].float().cpu().numpy()
        assert G.within_bound(y2, y_ref, bound, bf16_out=True).all()


def test_decode_forward_replays_as_a_cuda_graph():
    """The decode forward captured into a CUDA graph and replayed gives the
    eager forward's outputs bit for bit (every library call is capturable
    once its one-time setup has run), also after new activations are copied
    into the captured input buffer."""
    import torch
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    from precision_moe_numerics_nvfp4_gb300.pipeline import MoELayer
    m = W.decode("cuda")
    M, D, I, E = m.x_perm.shape[0], 7168, 2048, 128
    layer = MoELayer(M, D, I, E, backward=False)
    layer.quantize_weights(m.w13, m.w2)
    x = m.x_perm.clone()
    graph = MoELayer.capture(lambda: layer.forward_activations(x, m.group_offsets))
    x2 = (m.x_perm.float() * 0.5).to(x.dtype)
    for src in (m.x_perm, x2):
        layer.forward_activations(src, m.group_offsets)
        torch.cuda.synchronize()
        want = layer.y2.clone()
        layer.y2.zero_()
        x.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(layer.y2, want)
    assert N.nvfp4moe_get_device_status() == 0
