"""GPU parity of the quantization steps (amax -> outer scale, NVFP4 quantize,
the SR re-quantization to transposed MXFP8, the gradient MXFP8 quantizer)
against the oracle:
codes, scales (every byte of the scale buffer, padding included) and outer
scales must be bit-exact, stochastic rounding included for a given seed."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import layout as L
from oracle import mxfp8 as MX
from oracle import nvfp4 as NV
from oracle import requant as RQ
from oracle import swiglu as SW
from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
from precision_moe_numerics_nvfp4_gb300 import workloads as W
from tests.gpu_helpers import (bf16_f32, check_status, dev, filled, gempty, gfull, gpu_nvfp4, oracle_nvfp4,
                               unpack_gpu_nvfp4)

pytestmark = pytest.mark.gpu


def _tensor(shape, seed, kind="t", scale=0.05):
    g = torch.Generator(device="cuda").manual_seed(seed)
    if kind == "t":
        x = W.student_t(shape, 3, scale, g, "cuda")
        W.plant_elements(x, max(1, x.numel() // 1000), 1000.0, g)
    else:
        x = torch.randn(shape, generator=g, device="cuda") * scale
    return x.to(torch.bfloat16).contiguous()


def _groups(sizes):
    o = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    return torch.from_numpy(o).to(dev()), o


# ---- amax + NVFP4 quantize --------------------------------------------------------------
@pytest.mark.parametrize("batch,rows,cols", [(1, 256, 512), (1, 1024, 512), (1, 300, 272), (3, 200, 160),
                                             (1, 1, 16), (2, 129, 64)])
def test_nvfp4_quantize_matches_oracle(batch, rows, cols):
    x = _tensor((batch, rows, cols), seed=rows * 7 + cols)
    codes, scales, sg = gpu_nvfp4(x, batch, rows, cols)
    ec, es, esg = oracle_nvfp4(bf16_f32(x), batch, rows, cols)
    assert np.array_equal(sg.view(np.uint32), esg.view(np.uint32))
    assert np.array_equal(codes, ec)
    assert np.array_equal(scales, es)


def test_nvfp4_quantize_single_linear_workload():
    s = W.single_linear("cuda")
    for t in (s.x, s.w):
        r, c = t.shape
        codes, scales, sg = gpu_nvfp4(t.contiguous(), 1, r, c)
        ec, es, esg = oracle_nvfp4(bf16_f32(t), 1, r, c)
        assert sg[0] == esg[0] and np.array_equal(codes, ec) and np.array_equal(scales, es)


def _many_groups(n, seed):
    """n groups of 0..9 rows (many empty): more groups than the window
    lookup's first four chunks of 32."""
    return [int(v) for v in np.random.default_rng(seed).integers(0, 10, size=n)]


@pytest.mark.parametrize("sizes", [[5, 0, 295, 128, 272, 0], _many_groups(200, 1), _many_groups(300, 2)],
                         ids=["six", "200_groups", "300_groups"])
def test_nvfp4_quantize_grouped_layout(sizes):
    go, o = _groups(sizes)
    rows, cols = int(o[-1]), 256
    x = _tensor((rows, cols), seed=11)
    codes, scales, sg = gpu_nvfp4(x, 1, rows, cols, go)
    ec, es, esg = oracle_nvfp4(bf16_f32(x), 1, rows, cols, groups=o)
    assert sg[0] == esg[0] and np.array_equal(codes, ec) and np.array_equal(scales, es)


def test_nvfp4_page_examples_with_unit_outer_scale():
    # "Low-precision formats on Blackwell": a block whose largest value is -54
    # stores -6 with scale 9; 5.4 (bf16 5.40625) in it becomes 0.5 -> 4.5;
    # 592 (the bf16 neighbour of 593.7) gets scale 96 and code 6.
    x = torch.zeros((2, 16), dtype=torch.bfloat16, device=dev())
    x[0, 0], x[0, 1], x[1, 0] = -54.0, 5.4, 592.0
    one = torch.ones(1, dtype=torch.float32, device=dev())
    codes, scales, _ = gpu_nvfp4(x, 1, 2, 16, sg_in=one)
    c, s = unpack_gpu_nvfp4(codes, scales, 1, 2, 16)
    assert F.e4m3_decode(int(s[0, 0])) == 9.0 and F.e2m1_decode(int(c[0, 0])) == -6.0
    assert F.e2m1_decode(int(c[0, 1])) == 0.5
    assert F.e4m3_decode(int(s[1, 0])) == 96.0 and F.e2m1_decode(int(c[1, 0])) == 6.0


def test_nvfp4_zero_tensor_and_signed_zero():
    x = torch.zeros((128, 64), dtype=torch.bfloat16, device=dev())
    x[3, 5] = -0.0
    codes, scales, sg = gpu_nvfp4(x, 1, 128, 64)
    c, s = unpack_gpu_nvfp4(codes, scales, 1, 128, 64)
    assert sg[0] == 1.0 and np.all(s == 0) and c[3, 5] == 0x8 and np.count_nonzero(c) == 1


def test_nvfp4_cvt_rounding_sweep():
    """Every bf16 value times a scale-1 block: the hardware conversions (E4M3
    scale, E2M1 codes) agree with the oracle's brute-force rounding."""
    allbits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    vals = allbits.float()
    ok = torch.isfinite(vals) & (vals.abs() <= 2688.0)
    vals = vals[ok]
    vals = vals[: (vals.numel() // 16) * 16].reshape(-1, 16).to(torch.bfloat16).to(dev())
    sg = gfull((1,), 1.0, dtype=torch.float32, device=dev())
    r, c = vals.shape
    codes, scales, _ = gpu_nvfp4(vals.contiguous(), 1, r, c, sg_in=sg)
    ec, es, _ = oracle_nvfp4(bf16_f32(vals), 1, r, c, sg_in=[1.0])
    assert np.array_equal(codes, ec) and np.array_equal(scales, es)


def test_nvfp4_bad_offsets_recorded_and_nothing_written():
    go = torch.tensor([0, 10, 5, 40], dtype=torch.int32, device=dev())
    x = _tensor((40, 64), seed=3)
    cb, sb = N.nvfp4_sizes(1, 40, 64, 3)
    codes, scales = filled(cb), filled(sb)
    one = torch.ones(1, dtype=torch.float32, device=dev())
    N.nvfp4_quantize(x, 1, 40, 64, go, one, None, codes, scales, None)
    assert N.nvfp4moe_get_device_status() == N.NV_ERR_OFFSETS
    assert torch.all(codes == 0xA5) and torch.all(scales == 0xA5)
    assert N.nvfp4moe_get_device_status() == 0


@pytest.mark.parametrize("offsets", [[0, 10, 5, 40], [0, 10, 20, 39], [3, 10, 20, 40], [0, -1, 20, 40]],
                         ids=["decreasing", "last_not_rows", "first_not_zero", "negative"])
def test_bad_offsets_recorded_and_nothing_written_every_grouped_quantizer(offsets):
    """The group lookup of every grouped quantizer (NVFP4 quantize, the MXFP8
    gradient quantizer row-wise + transposed, the fused quantize + SR
    requant) rejects offsets that are not a partition of the rows: the status
    word says NV_ERR_OFFSETS and no output byte changes."""
    from precision_moe_numerics_nvfp4_gb300.pipeline import MxRows, MxTransposed, NvTensor
    go = torch.tensor(offsets, dtype=torch.int32, device=dev())
    R, C, E = 40, 128, 3
    x = _tensor((R, C), seed=5)
    one = torch.ones(1, dtype=torch.float32, device=dev())
    nv, mr, mt = NvTensor(1, R, C, dev(), E=E), MxRows(R, C, dev(), E=E), MxTransposed(R, C, dev(), E=E)
    outs = (nv.codes, nv.scales, mr.codes, mr.scales, mt.codes, mt.scales)
    for t in outs:
        t.fill_(0xA5)
    N.nvfp4_quantize(x, 1, R, C, go, one, None, nv.codes, nv.scales, None)
    assert N.nvfp4moe_get_device_status() == N.NV_ERR_OFFSETS
    N.mxfp8_quantize(x, R, C, go, N.NV_SR, 1, 2, 3, mr.codes, mr.scales, mt.codes, mt.scales)
    assert N.nvfp4moe_get_device_status() == N.NV_ERR_OFFSETS
    N.nvfp4_quantize_requant(x, 1, R, C, go, one, None, nv.codes, nv.scales, None, 1, 2, mt.codes, mt.scales)
    assert N.nvfp4moe_get_device_status() == N.NV_ERR_OFFSETS
    for t in outs:
        assert torch.all(t == 0xA5)
    assert N.nvfp4moe_get_device_status() == 0


def test_host_argument_errors():
    x = torch.zeros((4, 24), dtype=torch.bfloat16, device=dev())
    c = filled(64)
    with pytest.raises(N.NvError) as e:
        N.nvfp4_quantize(x, 1, 4, 24, None, None, None, c, c, None)
    assert e.value.status == N.NV_ERR_SHAPE
    x2 = torch.zeros((4, 32), dtype=torch.bfloat16, device=dev())
    with pytest.raises(N.NvError) as e:
        N.nvfp4_quantize(x2, 1, 4, 32, None, None, None, c, c, None)
    assert e.value.status == N.NV_ERR_WORKSPACE


def test_wait_timeout_is_reported_not_hung():
    N.nvfp4moe_selftest_wait_timeout(2000)
    assert N.nvfp4moe_get_device_status() == N.NV_ERR_TIMEOUT
    # the context is still usable
    test_nvfp4_quantize_matches_oracle(1, 1, 16)


# ---- MXFP8 row-wise and transposed -------------------------------------------------
def _gpu_mx(x, rows, cols, groups, mode, seed, off_row, off_t, want_row=True, want_t=True):
    E = None if groups is None else groups.numel() - 1
    out = {}
    cr = sr = ct = st = None
    if want_row:
        nb, sbts = N.mxfp8_row_sizes(rows, cols, E)
        cr, sr = filled(nb), filled(sbts)
    if want_t:
        P, nb, sbts = N.mxfp8_t_sizes(rows, cols, E)
        ct, st = filled(nb, 0), filled(sbts)
        out["P"] = P
    N.mxfp8_quantize(x, rows, cols, groups, mode, seed, off_row, off_t, cr, sr, ct, st)
    check_status()
    out.update(cr=cr, sr=sr, ct=ct, st=st)
    return {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in out.items()}


def _oracle_mx_row(xf, groups, mode, seed, off):
    rows, cols = xf.shape
    if mode == N.NV_SR:
        codes, sc = RQ.quantize_grad_rowwise(xf, seed, off)
    else:
        codes, sc = MX.quantize(xf, "rn")
    if groups is None:
        rmap, prow = np.arange(rows), L.roundup(rows, 128)
    else:
        rmap, prow = L.grouped_row_map(groups), L.padded_cap(rows, len(groups) - 1)
    return codes.reshape(-1), L.swizzle(sc, rmap, prow)


def _oracle_mx_t(xf, groups, mode, seed, off, P):
    rows, cols = xf.shape
    o = np.array([0, rows]) if groups is None else groups
    if mode == N.NV_SR:
        codes, sc = RQ.transposed_grouped_sr(xf, o, seed, off, P)
    else:
        raise NotImplementedError
    return codes, sc


@pytest.mark.parametrize("mode", [N.NV_RN, N.NV_SR])
@pytest.mark.parametrize("rows,cols,sizes", [(300, 256, None), (700, 128, [5, 0, 295, 128, 272]),
                                             (256, 1024, None)])
def test_mxfp8_rowwise_only(mode, rows, cols, sizes):
    x = _tensor((rows, cols), seed=rows + cols, kind="n", scale=1e-3)
    go, o = (None, None) if sizes is None else _groups(sizes)
    r = _gpu_mx(x, rows, cols, go, mode, 5, 2, 3, want_t=False)
    ec, es = _oracle_mx_row(bf16_f32(x), o, mode, 5, 2)
    assert np.array_equal(r["cr"], ec)
    assert np.array_equal(r["sr"], es)


@pytest.mark.parametrize("want_row", [False, True])
@pytest.mark.parametrize("rows,cols,sizes", [(700, 128, [5, 0, 295, 128, 272]), (256, 1024, None),
                                             (513, 256, [1, 512]), (None, 128, _many_groups(260, 3))])
def test_mxfp8_transposed_grouped_sr(want_row, rows, cols, sizes):
    if rows is None:
        rows = sum(sizes)
    x = _tensor((rows, cols), seed=rows * 3 + cols, kind="n", scale=1e-3)
    go, o = (None, None) if sizes is None else _groups(sizes)
    r = _gpu_mx(x, rows, cols, go, N.NV_SR, 9, 4, 5, want_row=want_row, want_t=True)
    xf = bf16_f32(x)
    ec, es = _oracle_mx_t(xf, o, N.NV_SR, 9, 5, r["P"])
    ogroups = np.array([0, rows]) if o is None else o
    Ptot = int(L.group_padded_starts(ogroups)[-1])
    gpu_codes = r["ct"].reshape(cols, r["P"])
    assert np.array_equal(gpu_codes[:, :Ptot], ec[:, :Ptot])
    gpu_sc = L.unswizzle(r["st"], np.arange(cols), r["P"] // 32)
    assert np.array_equal(gpu_sc, es)
    if want_row:
        ec2, es2 = _oracle_mx_row(xf, o, N.NV_SR, 9, 4)
        assert np.array_equal(r["cr"], ec2)
        assert np.array_equal(r["sr"], es2)


def test_mxfp8_single_linear_gradient():
    s = W.single_linear("cuda")
    g = s.g.contiguous()
    rows, cols = g.shape
    r = _gpu_mx(g, rows, cols, None, N.NV_SR, 0, 2, 3)
    gf = bf16_f32(g)
    ec, es = _oracle_mx_row(gf, None, N.NV_SR, 0, 2)
    assert np.array_equal(r["cr"], ec) and np.array_equal(r["sr"], es)
    tc, ts = _oracle_mx_t(gf, None, N.NV_SR, 0, 3, r["P"])
    assert np.array_equal(r["ct"].reshape(cols, r["P"]), tc)


# ---- dequant -> transpose -> SR requant ------------------------------------------
def _gpu_requant(codes, scales, sg, batch, rows, cols, groups, seed, off):
    if groups is None:
        nb, sbts = N.requant_weight_sizes(batch, rows, cols)
    else:
        _, nb, sbts = N.mxfp8_t_sizes(rows, cols, groups.numel() - 1)
    oc, os_ = filled(nb, 0), filled(sbts)
    N.dequant_transpose_requant_sr(codes, scales, sg, batch, rows, cols, groups, seed, off, oc, os_)
    check_status()
    return oc.cpu().numpy(), os_.cpu().numpy()


def _nvfp4_on_gpu(x, batch, rows, cols, groups=None):
    E = None if groups is None else groups.numel() - 1
    cb, sb = N.nvfp4_sizes(batch, rows, cols, E)
    codes, scales = filled(cb), filled(sb)
    sg = gempty(batch, dtype=torch.float32, device=dev())
    ws = filled(N.nvfp4moe_quantize_workspace_bytes(batch, rows, cols), 0)
    N.nvfp4_quantize(x, batch, rows, cols, groups, None, sg, codes, scales, ws)
    check_status()
    return codes, scales, sg


@pytest.mark.parametrize("batch,rows,cols", [(1, 1024, 512), (2, 256, 384), (1, 128, 128)])
def test_requant_weights_matches_oracle(batch, rows, cols):
    x = _tensor((batch, rows, cols), seed=batch * 100 + rows, kind="n", scale=0.02)
    codes, scales, sg = _nvfp4_on_gpu(x, batch, rows, cols)
    oc, os_ = _gpu_requant(codes, scales, sg, batch, rows, cols, None, 3, 0)
    c, s = unpack_gpu_nvfp4(codes.cpu().numpy(), scales.cpu().numpy(), batch, rows, cols)
    ec, es = RQ.requant_weights(c.reshape(batch, rows, cols), s.reshape(batch, rows, cols // 16), sg.cpu().numpy(),
                                3, 0)
    assert np.array_equal(oc.reshape(batch, cols, rows), ec)
    cpad = L.roundup(cols, 128)
    rmap = L.batched_row_map(batch, cols).reshape(batch, cols)
    assert cpad == cols
    got = L.unswizzle(os_, rmap.reshape(-1), rows // 32).reshape(batch, cols, rows // 32)
    assert np.array_equal(got, es)


@pytest.mark.parametrize("sizes,cols", [([5, 0, 295, 128, 272], 256), ([256], 512), ([1, 130, 0, 3], 128)])
def test_requant_grouped_activations_matches_oracle(sizes, cols):
    go, o = _groups(sizes)
    rows = int(o[-1])
    x = _tensor((rows, cols), seed=rows + 17, kind="n", scale=1.0)
    codes, scales, sg = _nvfp4_on_gpu(x, 1, rows, cols, go)
    oc, os_ = _gpu_requant(codes, scales, sg, 1, rows, cols, go, 7, 2)
    c, s = unpack_gpu_nvfp4(codes.cpu().numpy(), scales.cpu().numpy(), 1, rows, cols, o)
    P = N.nvfp4moe_padded_cap(rows, len(sizes))
    ec, es = RQ.requant_grouped(c, s, sg.cpu().numpy()[0], o, 7, 2, P)
    Ptot = int(L.group_padded_starts(o)[-1])
    assert np.array_equal(oc.reshape(cols, P)[:, :Ptot], ec[:, :Ptot])
    assert np.array_equal(L.unswizzle(os_, np.arange(cols), P // 32), es)


def test_quantizers_are_deterministic():
    x = _tensor((3, 256, 256), seed=42)
    a = gpu_nvfp4(x, 3, 256, 256)
    b = gpu_nvfp4(x, 3, 256, 256)
    assert all(np.array_equal(u, v) for u, v in zip(a, b))
    g = _tensor((700, 128), seed=43, kind="n")
    go, _ = _groups([5, 0, 295, 128, 272])
    r1 = _gpu_mx(g, 700, 128, go, N.NV_SR, 1, 2, 3)
    r2 = _gpu_mx(g, 700, 128, go, N.NV_SR, 1, 2, 3)
    assert all(np.array_equal(r1[k], r2[k]) for k in ("cr", "sr", "ct", "st"))


# ---- SwiGLU ----------------------------------------------------------------------------
def test_swiglu_forward_backward():
    M, I = 300, 1536
    y13 = _tensor((M, 2 * I), seed=5, kind="n", scale=1.0)
    dh = _tensor((M, I), seed=6, kind="n", scale=1e-3)
    h = gempty((M, I), dtype=torch.bfloat16, device=dev())
    d = gempty((M, 2 * I), dtype=torch.bfloat16, device=dev())
    N.nvfp4moe_swiglu_fwd(y13, M, I, h)
    N.nvfp4moe_swiglu_bwd(dh, y13, M, I, d)
    check_status()
    yf, dhf = bf16_f32(y13).astype(np.float64), bf16_f32(dh).astype(np.float64)
    href = SW.forward(yf)
    dref = SW.backward(dhf, yf)
    # fp32 math then one bf16 rounding: within 1 bf16 ulp of the float64 value
    for got, ref in ((bf16_f32(h), href), (bf16_f32(d), dref)):
        tol = np.abs(ref) * 2.0 ** -7 + 1e-30
        assert np.all(np.abs(got - ref) <= tol)


# ---- the quantization sweep at full size (sampled) -------------------------------------
@pytest.mark.parametrize("shape", W.QUANT_SWEEP_SHAPES)
def test_quant_sweep_full_size_sampled(shape):
    rows, cols = shape
    x = W.quant_sweep(shape, "cuda")
    codes, scales, sg = _nvfp4_on_gpu(x, 1, rows, cols)
    # outer scale from the whole tensor, exactly
    xf_all = bf16_f32(x)
    esg = NV.outer_scale(xf_all)
    assert sg.cpu().numpy()[0] == esg
    rng = np.random.default_rng(rows)
    out_rows = np.unique(np.concatenate([rng.choice(rows, 24, replace=False),
                                         np.nonzero(np.abs(xf_all).max(axis=1) > 10)[0][:8], [0, rows - 1]]))
    cpu_codes = codes.cpu().numpy().reshape(rows, cols // 2)
    cpu_scales = scales.cpu().numpy()
    for r in out_rows:
        ec, es, _ = NV.quantize(xf_all[r:r + 1], esg)
        assert np.array_equal(cpu_codes[r], NV.pack(ec)[0])
        got = L.unswizzle(cpu_scales, np.array([r]), cols // 16)
        assert np.array_equal(got, es)
    # MXFP8 RN along rows
    nb, sbts = N.mxfp8_row_sizes(rows, cols)
    mc, ms = filled(nb), filled(sbts)
    N.mxfp8_quantize(x, rows, cols, None, N.NV_RN, 0, 0, 0, mc, ms, None, None)
    check_status()
    mcn, msn = mc.cpu().numpy().reshape(rows, cols), ms.cpu().numpy()
    for r in out_rows[:12]:
        ec, es = MX.quantize(xf_all[r:r + 1], "rn")
        assert np.array_equal(mcn[r], ec[0])
        assert np.array_equal(L.unswizzle(msn, np.array([r]), cols // 32), es)
    # requant of the NVFP4 result: sampled output rows (= source columns)
    oc, os_ = _gpu_requant(codes, scales, sg, 1, rows, cols, None, 1, 0)
    oc = oc.reshape(cols, rows)
    c_all = NV.unpack(cpu_codes)
    s_all = L.unswizzle(cpu_scales, np.arange(rows), cols // 16)
    for c in rng.choice(cols, 6, replace=False):
        kb = c // 16
        col_codes = c_all[:, c]
        col_scale = s_all[:, kb]
        deq = (F.decode_e2m1_array(col_codes) * F.decode_e4m3_array(col_scale)).astype(np.float32) * np.float32(esg)
        deq = deq.astype(np.float32)[None, :]
        r = np.arange(rows, dtype=np.int64)
        u = RQ.pair_draws16(1, 0, (r - (r & 1)) * cols + c)
        bits = np.where(r & 1, RQ.bitrev16(u), u)[None, :]
        ec, es = MX.quantize(deq, "sr", bits)
        assert np.array_equal(oc[c], ec[0])
        assert np.array_equal(L.unswizzle(os_, np.array([c]), rows // 32), es)


def test_requant_zero_blocks_with_large_outer_scale():
    """Whole 32-row column blocks of zeros (signed) next to values whose outer
    scale exceeds 2: the zeros must stay signed zeros with scale code 0."""
    rows, cols = 256, 128
    x = _tensor((rows, cols), seed=77, kind="n", scale=3000.0)
    x[32:64, :] = 0.0
    x[40, 5] = -0.0
    codes, scales, sg = _nvfp4_on_gpu(x, 1, rows, cols)
    assert sg.cpu().numpy()[0] > 2.0
    oc, os_ = _gpu_requant(codes, scales, sg, 1, rows, cols, None, 5, 1)
    c, s = unpack_gpu_nvfp4(codes.cpu().numpy(), scales.cpu().numpy(), 1, rows, cols)
    ec, es = RQ.requant_weights(c[None], s[None], sg.cpu().numpy(), 5, 1)
    assert np.array_equal(oc.reshape(1, cols, rows), ec)
    got = L.unswizzle(os_, L.batched_row_map(1, cols), rows // 32).reshape(1, cols, rows // 32)
    assert np.array_equal(got, es)
    assert np.all(es[0, :, 1] == 0)


@pytest.mark.parametrize("mode", [N.NV_RN, N.NV_SR])
def test_mxfp8_wide_range_blocks_match_oracle(mode):
    """Blocks whose elements span the E4M3 subnormal range, the normal range
    and the saturation region (|w| in [416, 512)), with signed zeros: the
    hardware conversions agree with the oracle's rules everywhere."""
    rows, cols = 256, 256
    rng = np.random.default_rng(31)
    mag = np.exp2(rng.uniform(-16, 9, size=(rows, cols)))
    v = mag * rng.choice([-1.0, 1.0], size=(rows, cols))
    v[rng.random((rows, cols)) < 0.03] = 0.0
    v[rng.random((rows, cols)) < 0.01] = -0.0
    v[:, ::32] = np.where(rng.random((rows, cols // 32)) < 0.5, 256.0, -300.0)   # block maxima
    v[::7, 5] = 470.0                                                              # saturating elements
    x = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).to(dev()).contiguous()
    r = _gpu_mx(x, rows, cols, None, mode, 12, 3, 4, want_row=True, want_t=(mode == N.NV_SR))
    xf = bf16_f32(x)
    ec, es = _oracle_mx_row(xf, None, mode, 12, 3)
    assert np.array_equal(r["cr"], ec) and np.array_equal(r["sr"], es)
    if mode == N.NV_SR:
        tc, ts = _oracle_mx_t(xf, None, mode, 12, 4, r["P"])
        assert np.array_equal(r["ct"].reshape(cols, r["P"]), tc)
        assert np.array_equal(L.unswizzle(r["st"], np.arange(cols), r["P"] // 32), ts)
