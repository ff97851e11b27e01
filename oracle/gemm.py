"""FP64 references for the grouped expert GEMMs.  Test infrastructure only.

End-to-End 4-Bit Training, "Block-scaled backward passes": the forward pass
computes y = x_q w_q^T -- a dot product takes 16-value blocks from a row of x_q
and a column of w_q^T, multiplies the pairs and scales the sum by both block
scales -- and the backward pass computes dx = g w_q and dw = g^T x_q.
"Quantized communications": the tokens routed to an expert are computed by
that expert, so each expert e multiplies only its own rows (its group).

The reference is the exact product of the dequantized operands in float64
(numpy matmul is the library step); the accepted error is
|y - y_ref| <= 1e-4 * (|A| |B|)_ij element-wise, plus half a bf16 ulp of y_ref
when the output is bf16.
"""
from __future__ import annotations

import numpy as np

REL_BOUND = 1e-4


def grouped_rows(A64, B64, group_offsets):
    """y[o_e:o_{e+1}] = A64[o_e:o_{e+1}] @ B64[e].T for every group e.
    A64 [M, K], B64 [E, N, K].  Returns (y_ref [M, N], bound [M, N])."""
    A64 = np.asarray(A64, dtype=np.float64)
    B64 = np.asarray(B64, dtype=np.float64)
    o = np.asarray(group_offsets, dtype=np.int64)
    M = A64.shape[0]
    N = B64.shape[1]
    y = np.zeros((M, N))
    bound = np.zeros((M, N))
    for e in range(len(o) - 1):
        a = A64[o[e]:o[e + 1]]
        if a.shape[0] == 0:
            continue
        y[o[e]:o[e + 1]] = a @ B64[e].T
        bound[o[e]:o[e + 1]] = np.abs(a) @ np.abs(B64[e]).T
    return y, bound


def grouped_contraction(AT64, BT64, padded_starts):
    """Weight-gradient form: dw_e = AT64[:, cols_e] @ BT64[:, cols_e].T where
    cols_e is group e's padded token range [P_e, P_{e+1}).  AT64 [N, P],
    BT64 [K, P].  Returns (dw_ref [E, N, K], bound [E, N, K])."""
    AT64 = np.asarray(AT64, dtype=np.float64)
    BT64 = np.asarray(BT64, dtype=np.float64)
    P = np.asarray(padded_starts, dtype=np.int64)
    E = len(P) - 1
    N, K = AT64.shape[0], BT64.shape[0]
    dw = np.zeros((E, N, K))
    bound = np.zeros((E, N, K))
    for e in range(E):
        a = AT64[:, P[e]:P[e + 1]]
        b = BT64[:, P[e]:P[e + 1]]
        dw[e] = a @ b.T
        bound[e] = np.abs(a) @ np.abs(b).T
    return dw, bound


def bf16_half_ulp(y_ref) -> np.ndarray:
    """Half a unit in the last place of bf16 at |y_ref| (8 significant bits)."""
    a = np.abs(np.asarray(y_ref, dtype=np.float64))
    _, ex = np.frexp(np.where(a == 0, 1.0, a))
    half = np.ldexp(1.0, ex - 1 - 8)          # ulp = 2^(floor(log2 a) - 7)
    return np.where(a == 0, np.ldexp(1.0, -133), half)


def within_bound(y, y_ref, bound, bf16_out: bool = False, rel: float = REL_BOUND):
    """Boolean mask of elements that meet the bound."""
    err = np.abs(np.asarray(y, dtype=np.float64) - y_ref)
    lim = rel * bound
    if bf16_out:
        # the bf16 rounding of the fp32 result: half an ulp at the larger of
        # |y| and |y_ref| (they can straddle a power of two)
        lim = lim + bf16_half_ulp(np.maximum(np.abs(np.asarray(y, dtype=np.float64)), np.abs(y_ref)))
    return err <= lim
