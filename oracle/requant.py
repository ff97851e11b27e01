"""Backward-pass re-quantization: dequantize the forward NVFP4 tensor,
transpose it at higher precision, and stochastically re-quantize to MXFP8; and
the SR quantization of the BF16 output gradient, row-wise and transposed.
Test infrastructure only.

End-to-End 4-Bit Training, "Re-quantization with stochastic rounding": the
forward tensors are de-quantized, transposed in higher precision, then
re-quantized with SR so that E[w_q] = E[(w_q^T)^T]; re-quantizing to MXFP8 and
computing the gradients with MXFP8 GEMMs is the chosen trade-off.  Chinese
translation, Figure 4: saved weights and activations each go
dequantize -> transpose -> SR-quantize to MXFP8; the BF16 gradient is
SR-quantized to MXFP8 directly (DGRAD operand) and after a transpose (WGRAD
operand).

Conventions: "higher precision" is fp32 (the dequantized value
fp32(fp32(e2m1 * e4m3) * sg)); the random bits of every element are drawn from
its row-major index in the source tensor (see ``philox``), so they do not
depend on the transpose, the padding or the launch shape; the transposed
activations of each expert group are padded with zeros to a multiple of 128
tokens and placed at the group-padded column P_e (see ``layout``).
"""
from __future__ import annotations

import numpy as np

from . import layout as L
from . import mxfp8 as MX
from . import nvfp4 as NV
from .philox import element_bits16

F32 = np.float32


def _sr_bits(seed, offset, idx):
    return element_bits16(seed, offset, idx)


def requant_weights(codes, scales, sg, seed: int, offset: int):
    """Per-expert weights: NVFP4 codes [B, R, C] (4-bit codes), E4M3 scales
    [B, R, C/16], outer scales sg [B]  ->  MXFP8 (SR) of the transposes:
    E4M3 codes [B, C, R] and E8M0 scales [B, C, R/32].  R % 32 == 0.
    Element (b, r, c) draws the bits of index b*R*C + r*C + c."""
    codes = np.asarray(codes)
    B, R, C = codes.shape
    oc = np.empty((B, C, R), dtype=np.uint8)
    osc = np.empty((B, C, R // 32), dtype=np.uint8)
    for b in range(B):
        deq = NV.dequantize_f32(codes[b], scales[b], np.asarray(sg, dtype=F32).reshape(-1)[b])
        t = deq.T
        rr, cc = np.meshgrid(np.arange(R, dtype=np.int64), np.arange(C, dtype=np.int64), indexing="xy")
        idx = b * R * C + rr * C + cc           # [C, R] source index of T[c, r]
        oc[b], osc[b] = MX.quantize(t, "sr", _sr_bits(seed, offset, idx))
    return oc, osc


def transposed_grouped_sr(values, group_offsets, seed: int, offset: int, P_cols: int):
    """Transpose each expert group of a float32 matrix [M, C] to [C, M_e],
    zero-pad to M'_e = roundup(M_e, 128) columns, place it at column P_e of a
    [C, P_cols] matrix and SR-quantize to MXFP8 along the new rows.
    Element (m, c) draws the bits of source index m*C + c; padding is zero.
    Returns (E4M3 codes [C, P_cols], E8M0 scales [C, P_cols/32]); columns past
    the last group stay zero."""
    v = np.asarray(values, dtype=F32)
    M, C = v.shape
    o = np.asarray(group_offsets, dtype=np.int64)
    P = L.group_padded_starts(o)
    oc = np.zeros((C, P_cols), dtype=np.uint8)
    osc = np.zeros((C, P_cols // 32), dtype=np.uint8)
    for e in range(len(o) - 1):
        m0, m1 = int(o[e]), int(o[e + 1])
        Me = m1 - m0
        if Me == 0:
            continue
        Mp = L.roundup(Me, 128)
        t = np.zeros((C, Mp), dtype=F32)
        t[:, :Me] = v[m0:m1].T
        rows = np.arange(Mp, dtype=np.int64)[None, :]
        cols = np.arange(C, dtype=np.int64)[:, None]
        idx = np.where(rows < Me, (m0 + rows) * C + cols, 0)
        bits = np.where(rows < Me, _sr_bits(seed, offset, idx), 0)
        c_, s_ = MX.quantize(t, "sr", bits)
        oc[:, P[e]:P[e] + Mp] = c_
        osc[:, P[e] // 32:(P[e] + Mp) // 32] = s_
    return oc, osc


def requant_grouped(codes, scales, sg, group_offsets, seed: int, offset: int, P_cols: int):
    """Grouped activations: NVFP4 codes [M, C], E4M3 scales [M, C/16], one
    outer scale  ->  per-group transposed MXFP8 (SR) [C, P_cols]."""
    deq = NV.dequantize_f32(codes, scales, sg)
    return transposed_grouped_sr(deq, group_offsets, seed, offset, P_cols)


def quantize_grad_rowwise(g, seed: int, offset: int):
    """BF16 gradient [M, N] (as float32) -> MXFP8 with SR along rows.
    Element (m, n) draws the bits of index m*N + n."""
    g = np.asarray(g, dtype=F32)
    M, N = g.shape
    idx = np.arange(M * N, dtype=np.int64).reshape(M, N)
    return MX.quantize(g, "sr", _sr_bits(seed, offset, idx))


def quantize_rowwise_rn(v):
    """MXFP8 round-to-nearest along rows (the quantization-only sweep)."""
    return MX.quantize(np.asarray(v, dtype=F32), "rn")
