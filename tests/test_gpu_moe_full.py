"""Full-size, stage-wise parity of one MoE expert layer step (forward and
backward) at the benchmark workload: 16384 tokens x top-8 = 131072 rows,
d_model 4096, d_ff 1536, 64 experts with uneven groups.  The step runs exactly
as bench.py times it (the tokens and the routing map in, the routed rows
gathered by the quantization of x); afterwards sampled outputs of every stage are compared
with the oracle fed the GPU's own input to that stage:
codes / scales / outer scales bit-exact (stochastic rounding included), GEMM
outputs within 1e-4 (|A||B|) (+ half a bf16 ulp), SwiGLU within a bf16 ulp.
Sampled: the largest expert, the smallest non-empty one and two random ones;
their first, last and six random rows (or output rows / columns); for the
weight gradients, whole rows of dW (every column) of the largest and the
smallest non-empty expert.  Every buffer of the layer has a guard region
after its end, checked once the step has run."""
import numpy as np
import pytest
import torch

from oracle import gemm as G
from oracle import layout as L
from oracle import mxfp8 as MX
from oracle import nvfp4 as NV
from oracle import requant as RQ
from oracle import swiglu as SW
from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
from precision_moe_numerics_nvfp4_gb300 import pipeline as PL
from precision_moe_numerics_nvfp4_gb300 import workloads as W
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

D, I, E = 4096, 1536, 64
SEED = 3


def _np(t):
    return t.detach().cpu().numpy()


def _bf16_rows(t, rows):
    return t[torch.as_tensor(rows, device=t.device)].float().cpu().numpy()


def _amax_bf16(t):
    bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16) & 0x7FFF
    return np.array([int(bits.max()) << 16], dtype=np.uint32).view(np.float32)[0]


def _pair_bits(seed, off, key, second):
    u = RQ.pair_draws16(seed, off, key)
    return np.where(second, RQ.bitrev16(u), u)


@pytest.fixture(scope="module")
def run():
    torch.cuda.synchronize()
    m = W.moe("cuda", seed=2, with_grad=True, grad_seed=SEED)
    M = m.x_perm.shape[0]
    with pytest.MonkeyPatch.context() as mp:  # every buffer of the layer with a guard region
        mp.setattr(PL, "_u8", lambda n, dev: gh.guarded_bytes(max(int(n), 16)))
        mp.setattr(PL, "_empty", lambda shape, dtype, dev: gh.gempty(shape, dtype=dtype, device=dev))
        layer = PL.MoELayer(M, D, I, E)
    # the tokens and the routing map, as bench.py runs it: the quantization of
    # x gathers the routed rows (m.x_perm, which the oracle side reads)
    assert layer.gathers_rows
    layer.step(m.x, m.w13, m.w2, m.g2, m.group_offsets, seed=SEED, x_rows=m.rows)
    torch.cuda.synchronize()
    assert N.nvfp4moe_get_device_status() == 0
    gh.check_guards()
    gh.clear_guards()
    o = _np(m.group_offsets).astype(np.int64)
    sizes = np.diff(o)
    rng = np.random.default_rng(0)
    nonempty = np.nonzero(sizes)[0]
    experts = [int(np.argmax(sizes)), int(nonempty[np.argmin(sizes[nonempty])])]
    experts += [int(e) for e in rng.choice([e for e in nonempty if e not in experts], 2, replace=False)]
    rows = {}
    for e in experts:
        r = {int(o[e]), int(o[e + 1] - 1)}
        r |= set(int(v) for v in rng.integers(o[e], o[e + 1], size=6))
        rows[e] = sorted(r)
    return dict(m=m, layer=layer, o=o, M=M, experts=experts, rows=rows, rng=rng,
                rmap=L.grouped_row_map(o), P=L.group_padded_starts(o))


def _nv_rows(t, rows, rmap):
    """NVFP4 grouped tensor: 4-bit codes and E4M3 scales of the given rows."""
    C = t.cols
    codes = t.codes[: t.rows * C // 2].view(t.rows, C // 2)
    c = NV.unpack(_np(codes[torch.as_tensor(rows, device=codes.device)]))
    s = L.unswizzle(_np(t.scales), rmap[rows], C // 16)
    return c, s


def _nv_expert(t, e):
    """NVFP4 stacked weights: codes and scales of expert e."""
    R, C = t.rows, t.cols
    codes = t.codes[: t.batch * R * C // 2].view(t.batch, R, C // 2)[e]
    c = NV.unpack(_np(codes))
    s = L.unswizzle(_np(t.scales), e * L.roundup(R, 128) + np.arange(R), C // 16)
    return c, s, _np(t.sg)[e]


def _mx_rows(codes, scales, rows, C, rmap):
    cc = codes[: len(rmap) * C].view(len(rmap), C)[torch.as_tensor(rows, device=codes.device)]
    return _np(cc), L.unswizzle(_np(scales), rmap[rows], C // 32)


def _mx_t_row(t, c, P_cap):
    codes = _np(t.codes[c * P_cap:(c + 1) * P_cap])
    return codes, L.unswizzle(_np(t.scales), np.array([c]), P_cap // 32)[0]


def _mx_w_expert(t, e, R_out, C_out):
    """Transposed weights [E][R_out][C_out]: codes and scales of expert e."""
    codes = t.codes[: E * R_out * C_out].view(E, R_out, C_out)[e]
    s = L.unswizzle(_np(t.scales), e * L.roundup(R_out, 128) + np.arange(R_out), C_out // 32)
    return _np(codes), s


# ---- forward ---------------------------------------------------------------------
def test_forward_quantizers(run):
    m, layer, o = run["m"], run["layer"], run["o"]
    sg = _np(layer.xq.sg)[0]
    assert sg == NV.outer_scale(np.array([_amax_bf16(m.x_perm)], dtype=np.float32))
    sgh = _np(layer.hq.sg)[0]
    assert sgh == NV.outer_scale(np.array([_amax_bf16(layer.h)], dtype=np.float32))
    for e, rows in run["rows"].items():
        for t, src, s_ in ((layer.xq, m.x_perm, sg), (layer.hq, layer.h, sgh)):
            gc, gs = _nv_rows(t, rows, run["rmap"])
            ec, es, _ = NV.quantize(_bf16_rows(src, rows), s_)
            assert np.array_equal(gc, ec) and np.array_equal(gs, es)
    e = run["experts"][0]
    for t, w in ((layer.w13q, m.w13), (layer.w2q, m.w2)):
        gc, gs, gsg = _nv_expert(t, e)
        ec, es, esg = NV.quantize(w[e].float().cpu().numpy())
        assert gsg == esg and np.array_equal(gc, ec) and np.array_equal(gs, es)


def test_forward_gemms_and_swiglu(run):
    layer = run["layer"]
    for e, rows in run["rows"].items():
        xc, xs = _nv_rows(layer.xq, rows, run["rmap"])
        wc, ws, wsg = _nv_expert(layer.w13q, e)
        y_ref, bound = G.grouped_rows(NV.dequantize_f64(xc, xs, _np(layer.xq.sg)[0]),
                                      NV.dequantize_f64(wc, ws, wsg)[None], np.array([0, len(rows)]))
        y13 = _bf16_rows(layer.y13, rows)
        assert G.within_bound(y13, y_ref, bound, bf16_out=True).all()
        h_ref = SW.forward(y13.astype(np.float64))
        h = _bf16_rows(layer.h, rows)
        assert np.all(np.abs(h - h_ref) <= np.abs(h_ref) * 2.0 ** -7 + 1e-30)
        hc, hs = _nv_rows(layer.hq, rows, run["rmap"])
        w2c, w2s, w2sg = _nv_expert(layer.w2q, e)
        y_ref, bound = G.grouped_rows(NV.dequantize_f64(hc, hs, _np(layer.hq.sg)[0]),
                                      NV.dequantize_f64(w2c, w2s, w2sg)[None], np.array([0, len(rows)]))
        assert G.within_bound(_bf16_rows(layer.y2, rows), y_ref, bound, bf16_out=True).all()


# ---- backward: re-quantization and gradient quantization ----------------------------
def test_weight_requant(run):
    layer, rng = run["layer"], run["rng"]
    for t_nv, t_mx, off in ((layer.w13q, layer.w13t, PL.OFF_W13), (layer.w2q, layer.w2t, PL.OFF_W2)):
        R, C = t_nv.rows, t_nv.cols
        e = run["experts"][0]
        wc, ws, wsg = _nv_expert(t_nv, e)
        deq = NV.dequantize_f32(wc, ws, wsg)
        gcodes, gscales = _mx_w_expert(t_mx, e, C, R)
        for c in rng.choice(C, 4, replace=False):
            r = np.arange(R, dtype=np.int64)
            bits = _pair_bits(SEED, off, (e * R + r - (r & 1)) * C + c, (r & 1) == 1)
            ec, es = MX.quantize(deq[:, c][None], "sr", bits[None])
            assert np.array_equal(gcodes[c], ec[0]) and np.array_equal(gscales[c], es[0])


def _check_transposed(run, t_mx, values_of_group, C, off):
    """Transposed MXFP8 output rows c for the sampled experts' column ranges."""
    o, P = run["o"], run["P"]
    P_cap = t_mx.P
    for c in run["rng"].choice(C, 3, replace=False):
        gcodes, gscales = _mx_t_row(t_mx, c, P_cap)
        for e in run["experts"]:
            Me = int(o[e + 1] - o[e])
            Mp = L.roundup(Me, 128)
            v = np.zeros(Mp, dtype=np.float32)
            v[:Me] = values_of_group(e, c)
            t = np.arange(Mp, dtype=np.int64)
            bits = np.where(t < Me, _pair_bits(SEED, off, (o[e] + t - (t & 1)) * C + c, (t & 1) == 1), 0)
            ec, es = MX.quantize(v[None], "sr", bits[None])
            assert np.array_equal(gcodes[P[e]:P[e] + Mp], ec[0])
            assert np.array_equal(gscales[P[e] // 32:(P[e] + Mp) // 32], es[0])


def test_activation_requant(run):
    layer, o = run["layer"], run["o"]
    for t_nv, t_mx, C, off in ((layer.xq, layer.xt, D, PL.OFF_XQ), (layer.hq, layer.ht, I, PL.OFF_HQ)):
        sg = _np(t_nv.sg)[0]
        cache = {}

        def values(e, c, t_nv=t_nv, sg=sg, cache=cache):
            if e not in cache:
                rows = np.arange(o[e], o[e + 1])
                gc, gs = _nv_rows(t_nv, rows, run["rmap"])
                cache[e] = NV.dequantize_f32(gc, gs, sg)
            return cache[e][:, c]
        _check_transposed(run, t_mx, values, C, off)


def test_gradient_quantization(run):
    m, layer, o = run["m"], run["layer"], run["o"]
    for src, rowq, tq, C, off_r, off_t in ((m.g2, layer.g2_row, layer.g2t, D, PL.OFF_G2_ROW, PL.OFF_G2_T),
                                           (layer.dy13, layer.dy13_row, layer.dy13t, 2 * I, PL.OFF_DY13_ROW,
                                            PL.OFF_DY13_T)):
        for e, rows in run["rows"].items():
            gc, gs = _mx_rows(rowq.codes, rowq.scales, rows, C, run["rmap"])
            v = _bf16_rows(src, rows)
            rr = np.asarray(rows, dtype=np.int64)[:, None]
            n = np.arange(C, dtype=np.int64)[None, :]
            bits = _pair_bits(SEED, off_r, (rr * C + n - (n & 1)) // 2, (n & 1) == 1)
            ec, es = MX.quantize(v, "sr", bits)
            assert np.array_equal(gc, ec) and np.array_equal(gs, es)
        cache = {}

        def values(e, c, src=src, cache=cache):
            if e not in cache:
                cache[e] = _bf16_rows(src, np.arange(o[e], o[e + 1]))
            return cache[e][:, c]
        _check_transposed(run, tq, values, C, off_t)


# ---- backward GEMMs and SwiGLU backward --------------------------------------------
def test_backward_gemms_and_swiglu(run):
    layer, o, P, M = run["layer"], run["o"], run["P"], run["M"]
    # the step applied the SwiGLU backward in the w2 dgrad's epilogue (dh never
    # stored): it must equal the dgrad's bf16 dh followed by the SwiGLU
    # backward kernel, over the whole tensor
    assert layer.fuse_swiglu_bwd and layer.dh is None
    dh_full = gh.gempty((M, I), dtype=torch.bfloat16, device=gh.dev())
    dy13_ref = gh.gempty((M, 2 * I), dtype=torch.bfloat16, device=gh.dev())
    go = run["m"].group_offsets
    N.grouped_gemm_mxfp8_dx(layer.g2_row.codes, layer.g2_row.scales, layer.w2t.codes, layer.w2t.scales, go, E, M, D,
                            I, dh_full, N.NV_OUT_BF16)
    N.nvfp4moe_swiglu_bwd(dh_full, layer.y13, M, I, dy13_ref)
    torch.cuda.synchronize()
    assert N.nvfp4moe_get_device_status() == 0
    assert torch.equal(dy13_ref.view(torch.int16), layer.dy13.view(torch.int16))
    for e, rows in run["rows"].items():
        # dh = g2 w2 (dgrad of the down projection)
        gc, gs = _mx_rows(layer.g2_row.codes, layer.g2_row.scales, rows, D, run["rmap"])
        wc, ws = _mx_w_expert(layer.w2t, e, I, D)
        ref, bound = G.grouped_rows(MX.dequantize_f64(gc, gs), MX.dequantize_f64(wc, ws)[None],
                                    np.array([0, len(rows)]))
        dh = _bf16_rows(dh_full, rows)
        assert G.within_bound(dh, ref, bound, bf16_out=True).all()
        # dy13 = SwiGLU backward
        y13 = _bf16_rows(layer.y13, rows).astype(np.float64)
        d_ref = SW.backward(dh.astype(np.float64), y13)
        d = _bf16_rows(layer.dy13, rows)
        assert np.all(np.abs(d - d_ref) <= np.abs(d_ref) * 2.0 ** -7 + 1e-30)
        # dx = dy13 w13 (dgrad of gate/up)
        gc, gs = _mx_rows(layer.dy13_row.codes, layer.dy13_row.scales, rows, 2 * I, run["rmap"])
        wc, ws = _mx_w_expert(layer.w13t, e, D, 2 * I)
        ref, bound = G.grouped_rows(MX.dequantize_f64(gc, gs), MX.dequantize_f64(wc, ws)[None],
                                    np.array([0, len(rows)]))
        assert G.within_bound(_bf16_rows(layer.dx, rows), ref, bound, bf16_out=True).all()
    # weight gradients: whole rows dw[e][n][:] of the largest and the smallest
    # non-empty expert (first, last and two random rows), over the expert's
    # padded tokens
    rng = run["rng"]
    for gt, xt, dw, Nn, Kk in ((layer.g2t, layer.ht, layer.dw2, D, I), (layer.dy13t, layer.xt, layer.dw13, 2 * I, D)):
        P_cap = gt.P
        for e in run["experts"][:2]:
            cols = slice(P[e], P[e + 1])
            # B = x_q^T over the expert's tokens, all Kk rows: [Kk, P_e]
            b_c = _np(xt.codes[: Kk * P_cap].view(Kk, P_cap)[:, P[e]:P[e + 1]])
            b_s = L.unswizzle(_np(xt.scales), np.arange(Kk), P_cap // 32)[:, P[e] // 32:P[e + 1] // 32]
            b = MX.dequantize_f64(b_c, b_s)
            for n in sorted({0, Nn - 1} | set(int(v) for v in rng.choice(Nn, 2, replace=False))):
                a_c, a_s = _mx_t_row(gt, n, P_cap)
                a = MX.dequantize_f64(a_c[None, cols], a_s[None, P[e] // 32:P[e + 1] // 32])[0]
                ref = b @ a
                bound = np.abs(b) @ np.abs(a)
                got = _np(dw[e, int(n)]).astype(np.float64)
                assert np.all(np.abs(got - ref) <= 1e-4 * bound), (e, n)
