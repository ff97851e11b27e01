"""Pins of the oracle's GEMM references and SwiGLU: a hand-computed single
block, brute-force triple loops on tiny shapes, routing of rows to experts,
the bound's behaviour, and finite differences for the SwiGLU backward."""
import numpy as np

from oracle import formats as F
from oracle import gemm as G
from oracle import layout as L
from oracle import nvfp4 as NV
from oracle import swiglu as S


def test_single_block_by_hand():
    # "Block-scaled backward passes": a dot product takes 16-value blocks from
    # a row of x_q and a column of w_q^T, multiplies the pairs, sums, and
    # multiplies the sum by the scale of each block.
    a_codes = np.array([[0x1, 0x2, 0x3, 0x4, 0x5, 0x6, 0x7, 0x9, 0, 0, 0, 0, 0, 0, 0, 0xF]], dtype=np.uint8)
    b_codes = np.array([[0x2] * 16], dtype=np.uint8)
    a_scale = np.array([[0x40]], dtype=np.uint8)   # E4M3 2.0
    b_scale = np.array([[0x30]], dtype=np.uint8)   # E4M3 0.5
    # pairs: (0.5+1+1.5+2+3+4+6-0.5-6) * 1.0 = 11.5 ; times 2.0 * 0.5 ; times sg 1*1
    A = NV.dequantize_f64(a_codes, a_scale, 1.0)
    B = NV.dequantize_f64(b_codes, b_scale, 1.0)
    y, bound = G.grouped_rows(A, B[None], np.array([0, 1]))
    assert F.e4m3_decode(0x40) == 2.0 and F.e4m3_decode(0x30) == 0.5
    assert y[0, 0] == 11.5
    assert bound[0, 0] == (0.5 + 1 + 1.5 + 2 + 3 + 4 + 6 + 0.5 + 6)


def test_grouped_rows_brute_force():
    rng = np.random.default_rng(0)
    o = np.array([0, 3, 3, 7, 9])
    A = rng.standard_normal((9, 5))
    B = rng.standard_normal((4, 6, 5))
    y, bound = G.grouped_rows(A, B, o)
    for e in range(4):
        for i in range(o[e], o[e + 1]):
            for j in range(6):
                s = sum(A[i, k] * B[e, j, k] for k in range(5))
                t = sum(abs(A[i, k] * B[e, j, k]) for k in range(5))
                assert abs(y[i, j] - s) < 1e-12 and abs(bound[i, j] - t) < 1e-12


def test_rows_go_to_their_expert():
    o = np.array([0, 2, 5, 6])
    A = np.ones((6, 4))
    B = np.stack([np.full((3, 4), e + 1.0) for e in range(3)])
    y, _ = G.grouped_rows(A, B, o)
    assert np.all(y[0:2] == 4) and np.all(y[2:5] == 8) and np.all(y[5] == 12)


def test_grouped_contraction_brute_force():
    rng = np.random.default_rng(1)
    o = np.array([0, 130, 130, 140])
    P = L.group_padded_starts(o)
    AT = np.zeros((3, P[-1]))
    BT = np.zeros((2, P[-1]))
    g = rng.standard_normal((140, 3))
    x = rng.standard_normal((140, 2))
    for e in range(3):
        n = o[e + 1] - o[e]
        AT[:, P[e]:P[e] + n] = g[o[e]:o[e + 1]].T
        BT[:, P[e]:P[e] + n] = x[o[e]:o[e + 1]].T
    dw, bound = G.grouped_contraction(AT, BT, P)
    for e in range(3):
        ref = g[o[e]:o[e + 1]].T @ x[o[e]:o[e + 1]]
        assert np.allclose(dw[e], ref, rtol=0, atol=1e-12)
    assert np.all(dw[1] == 0)


def test_bound_accepts_and_rejects():
    y_ref = np.array([[1.0, -2.0, 0.0]])
    bound = np.array([[10.0, 10.0, 10.0]])
    ok = G.within_bound(y_ref + 0.9e-3, y_ref, bound)
    assert ok.all()
    bad = G.within_bound(y_ref + 1.1e-3, y_ref, bound)
    assert not bad.any()
    # bf16 output: half an ulp of the result is allowed on top
    assert G.within_bound(np.array([[1.0 + 2 ** -9, -2.0, 0.0]]), y_ref, bound * 0, bf16_out=True).all()
    assert not G.within_bound(np.array([[1.0 + 2 ** -7, -2.0, 0.0]]), y_ref, bound * 0, bf16_out=True)[0, 0]


def test_swiglu_forward_values():
    y13 = np.array([[0.0, 1.0, 3.0, 2.0], [-30.0, 30.0, 1.0, 1.0]])
    h = S.forward(y13)
    assert h[0, 0] == 0.0
    assert abs(h[0, 1] - (1 / (1 + np.exp(-1.0))) * 2.0) < 1e-15
    assert abs(h[1, 0]) < 1e-11 and abs(h[1, 1] - 30.0) < 1e-10


def test_swiglu_backward_finite_differences():
    rng = np.random.default_rng(2)
    y13 = rng.standard_normal((4, 8))
    dh = rng.standard_normal((4, 4))
    d = S.backward(dh, y13)
    eps = 1e-6
    num = np.zeros_like(y13)
    for i in range(4):
        for j in range(8):
            p = y13.copy(); p[i, j] += eps
            m = y13.copy(); m[i, j] -= eps
            num[i, j] = ((S.forward(p) - S.forward(m)) * dh).sum() / (2 * eps)
    assert np.allclose(d, num, rtol=1e-6, atol=1e-8)
