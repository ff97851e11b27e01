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
fp32(fp32(e2m1 * e4m3) * sg)); the transposed activations of each expert group
are padded with zeros to a multiple of 128 tokens and placed at the
group-padded column P_e (see ``layout``).  Random draws (see ``philox``) are
shared by the two elements of an output pair, the second using the draw
bit-reversed; the pair key comes from the source coordinates (r, c) of the
pair's first element in a source with C columns:
  * row-wise outputs (blocks along source rows, pairs (c, c+1), c even):
        K = (r * C + c) / 2
  * transposed outputs (blocks along source columns, pairs of source rows
    (r, r+1) at even positions of the output row):
        K = r * C + c
so the draws depend on the source positions and the pairing, not on the
launch shape; padding never draws.
"""
from __future__ import annotations

import numpy as np

from . import layout as L
from . import mxfp8 as MX
from . import nvfp4 as NV
from .philox import bitrev16, pair_draws16

F32 = np.float32


def _pair_bits(seed, offset, key, second):
    """Draw of each element: U(key) for the first element of its pair,
    bitrev16(U(key)) for the second."""
    u = pair_draws16(seed, offset, key)
    return np.where(second, bitrev16(u), u)


def requant_weights(codes, scales, sg, seed: int, offset: int, b0: int = 0):
    """Per-expert weights: NVFP4 codes [B, R, C] (4-bit codes), E4M3 scales
    [B, R, C/16], outer scales sg [B]  ->  MXFP8 (SR) of the transposes:
    E4M3 codes [B, C, R] and E8M0 scales [B, C, R/32].  R % 32 == 0.
    Output element (b, c, r) belongs to the pair of source rows (r0, r0+1),
    r0 = r - r % 2, with key ((b0 + b)*R + r0) * C + c; b0 > 0 treats the
    arrays as experts b0, b0+1, ... of a larger stack."""
    codes = np.asarray(codes)
    B, R, C = codes.shape
    oc = np.empty((B, C, R), dtype=np.uint8)
    osc = np.empty((B, C, R // 32), dtype=np.uint8)
    rr, cc = np.meshgrid(np.arange(R, dtype=np.int64), np.arange(C, dtype=np.int64), indexing="xy")  # [C, R]
    for b in range(B):
        deq = NV.dequantize_f32(codes[b], scales[b], np.asarray(sg, dtype=F32).reshape(-1)[b])
        key = ((b0 + b) * R + (rr - (rr & 1))) * C + cc
        bits = _pair_bits(seed, offset, key, (rr & 1) == 1)
        oc[b], osc[b] = MX.quantize(deq.T, "sr", bits)
    return oc, osc


def transposed_grouped_sr(values, group_offsets, seed: int, offset: int, P_cols: int):
    """Transpose each expert group of a float32 matrix [M, C] to [C, M_e],
    zero-pad to M'_e = roundup(M_e, 128) columns, place it at column P_e of a
    [C, P_cols] matrix and SR-quantize to MXFP8 along the new rows.
    Output element (c, t) of group e (token t, source row o_e + t) belongs to
    the pair of tokens (t0, t0+1), t0 = t - t % 2, with key (o_e + t0) * C + c;
    padding is zero.  Returns (E4M3 codes [C, P_cols], E8M0 scales
    [C, P_cols/32]); columns past the last group stay zero."""
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
        toks = np.arange(Mp, dtype=np.int64)[None, :]
        cols = np.arange(C, dtype=np.int64)[:, None]
        key = (m0 + toks - (toks & 1)) * C + cols
        bits = np.where(toks < Me, _pair_bits(seed, offset, key, (toks & 1) == 1), 0)
        c_, s_ = MX.quantize(t, "sr", bits)
        oc[:, P[e]:P[e] + Mp] = c_
        osc[:, P[e] // 32:(P[e] + Mp) // 32] = s_
    return oc, osc


def requant_grouped(codes, scales, sg, group_offsets, seed: int, offset: int, P_cols: int):
    """Grouped activations: NVFP4 codes [M, C], E4M3 scales [M, C/16], one
    outer scale  ->  per-group transposed MXFP8 (SR) [C, P_cols]."""
    deq = NV.dequantize_f32(codes, scales, sg)
    return transposed_grouped_sr(deq, group_offsets, seed, offset, P_cols)


def requant_grouped_rows(codes, scales, sg_rows, group_offsets, seed: int, offset: int, P_cols: int):
    """Grouped activations with per-token outer scales: the dequantized value
    of row r is fp32(fp32(e2m1 * e4m3) * sg_r); the rest as requant_grouped."""
    deq = NV.dequantize_rows_f32(codes, scales, sg_rows)
    return transposed_grouped_sr(deq, group_offsets, seed, offset, P_cols)


def quantize_grad_rowwise(g, seed: int, offset: int):
    """BF16 gradient [M, N] (as float32) -> MXFP8 with SR along rows.
    Element (m, n) belongs to the pair of columns (n0, n0+1), n0 = n - n % 2,
    with key (m*N + n0) / 2."""
    g = np.asarray(g, dtype=F32)
    M, N = g.shape
    mm, nn = np.meshgrid(np.arange(M, dtype=np.int64), np.arange(N, dtype=np.int64), indexing="ij")
    key = (mm * N + (nn - (nn & 1))) // 2
    return MX.quantize(g, "sr", _pair_bits(seed, offset, key, (nn & 1) == 1))


def quantize_rowwise_rn(v):
    """MXFP8 round-to-nearest along rows (the quantization-only sweep)."""
    return MX.quantize(np.asarray(v, dtype=F32), "rn")
