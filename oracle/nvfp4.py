"""NVFP4 block quantization (E2M1 values, one E4M3 scale per 1x16 block, one
FP32 outer scale per tensor).  Test infrastructure only.

End-to-End 4-Bit Training, "Low-precision formats on Blackwell": each block of
16 consecutive values is scaled by its largest magnitude -- a block whose
largest value is -54 stores -6 with scale 9 -- and a second FP32 scale over a
very large group (a whole tensor) shifts the representable range, so that a
value decodes as x_i^FP4 * x_{i//16}^FP8 * x^FP32.  "Recipe details": weights
use one outer scale per expert, i.e. each expert's matrix is "the tensor".

Conventions (the pages do not state them):
  sg       = fp32(amax / 2688) with 2688 = 6 * 448, or 1 when amax == 0
  den6     = fp32(6 * sg)
  s        = RN_E4M3(fp32(bamax / den6))          (saturates at 448)
  s == 0  -> every code is a signed zero, scale byte 0x00
  inv      = fp32(1 / fp32(s * sg))
  q_i      = RN_E2M1(fp32(x_i * inv))
  packing  : element 2j in the low nibble of byte j, 2j+1 in the high nibble
The element step multiplies by a per-block reciprocal rather than dividing.
Results are defined while s * sg is a normal fp32 number (any tensor whose
largest magnitude is at least 2^-100).

Per-token outer scales ("Recipe details": activations get one FP32 scale per
token, weights one per expert, for batch invariance): row r of an activation
matrix takes sg_r = fp32(amax_r / 2688) (1 for an all-zero row) and is
quantized exactly as a one-row tensor would be; dequantization multiplies by
its own sg_r.

Four Over Six (``quantize_four_over_six``): parity unpinned as to the
selection rule, which the pages do not give ("selects between two scale
factors"); the function states a reading and its pins check that reading.
"""
from __future__ import annotations

import numpy as np

from . import formats as F

F32 = np.float32
NVFP4_BLOCK = 16
OUTER_DEN = F32(6.0 * 448.0)  # 2688


def outer_scale(x) -> np.float32:
    """Per-tensor FP32 outer scale sg = amax / (6 * 448), or 1 for an
    all-zero tensor."""
    x = np.asarray(x, dtype=F32)
    amax = F32(np.max(np.abs(x))) if x.size else F32(0.0)
    if amax == 0:
        return F32(1.0)
    return F32(amax / OUTER_DEN)


def _quantize_blocks(xb: np.ndarray, sg, top: float = 6.0):
    """Quantize rows of a [nblocks, blocksize] float32 array, one scale each;
    ``sg`` is the outer scale, a scalar or one value per block; ``top`` is the
    E2M1 value the block maximum maps to (6; 4 for the Four Over Six
    candidate).  Returns (nibble codes [nblocks, blocksize], E4M3 scale codes
    [nblocks])."""
    sg = np.asarray(sg, dtype=F32)
    den6 = (F32(top) * sg).astype(F32)
    bamax = np.max(np.abs(xb), axis=1).astype(F32)
    s_code = F.rn_code((bamax / den6).astype(F32), F.E4M3_TABLE)
    s = F.decode_e4m3_array(s_code).astype(F32)
    nonzero = s != 0
    prod = (s * sg).astype(F32)
    with np.errstate(divide="ignore"):
        inv = np.where(nonzero, (F32(1.0) / np.where(nonzero, prod, F32(1.0))).astype(F32), F32(0.0))
    scaled = (xb * inv[:, None]).astype(F32)
    codes = F.rn_code(scaled, F.E2M1_TABLE)
    # an all-zero (or underflowed) block: signed zeros whatever the values
    zero_codes = np.where(np.signbit(xb), F.E2M1_SIGN, np.uint8(0)).astype(np.uint8)
    codes = np.where(nonzero[:, None], codes, zero_codes)
    return codes.astype(np.uint8), s_code.astype(np.uint8)


def quantize(x, sg=None):
    """NVFP4 1x16 round-to-nearest quantization of a float32 matrix [R, C]
    (C a multiple of 16) with blocks along the row.

    Returns (codes uint8 [R, C] of 4-bit E2M1 codes, scales uint8 [R, C/16]
    of E4M3 codes, sg float32).  ``sg`` defaults to ``outer_scale(x)``."""
    x = np.asarray(x, dtype=F32)
    R, C = x.shape
    if C % NVFP4_BLOCK:
        raise ValueError("C must be a multiple of 16")
    sg = outer_scale(x) if sg is None else F32(sg)
    codes, scales = _quantize_blocks(x.reshape(R * C // 16, 16), sg)
    return codes.reshape(R, C), scales.reshape(R, C // 16), sg


def outer_scale_rows(x) -> np.ndarray:
    """Per-token outer scales: sg_r = amax_r / 2688 of each row, 1 for an
    all-zero row (float32 [R])."""
    x = np.asarray(x, dtype=F32)
    amax = np.max(np.abs(x), axis=1).astype(F32) if x.shape[1] else np.zeros(x.shape[0], F32)
    return np.where(amax == 0, F32(1.0), (amax / OUTER_DEN).astype(F32)).astype(F32)


def quantize_rows(x, sg_rows=None):
    """NVFP4 1x16 RN quantization with one outer scale per row (per token).
    Returns (codes [R, C], scales [R, C/16], sg_rows float32 [R]);
    ``sg_rows`` defaults to ``outer_scale_rows(x)``."""
    x = np.asarray(x, dtype=F32)
    R, C = x.shape
    if C % NVFP4_BLOCK:
        raise ValueError("C must be a multiple of 16")
    sg_rows = outer_scale_rows(x) if sg_rows is None else np.asarray(sg_rows, dtype=F32).reshape(R)
    per_block = np.repeat(sg_rows, C // NVFP4_BLOCK)
    codes, scales = _quantize_blocks(x.reshape(R * C // 16, 16), per_block)
    return codes.reshape(R, C), scales.reshape(R, C // 16), sg_rows


def block_sq_error_f32(xb, codes, s_code, sg) -> np.ndarray:
    """Squared error of quantized blocks in fp32, in a fixed order: with the
    dequantized d_i = fp32(fp32(e2m1_i * s) * sg), e_i = fp32(x_i - d_i), the
    sum ((e_0^2 + e_1^2) + e_2^2) + ... over the block, each square and sum
    rounded to fp32.  [nblocks, 16] -> [nblocks]."""
    xb = np.asarray(xb, dtype=F32)
    q = F.decode_e2m1_array(codes)
    s = F.decode_e4m3_array(s_code)[:, None]
    d = ((q * s).astype(F32) * np.asarray(sg, dtype=F32).reshape(-1, 1)).astype(F32)
    e = (xb - d).astype(F32)
    sq = (e * e).astype(F32)
    acc = np.zeros(xb.shape[0], dtype=F32)
    for i in range(xb.shape[1]):
        acc = (acc + sq[:, i]).astype(F32)
    return acc


def quantize_four_over_six(x, sg=None, return_choice=False):
    """Four Over Six ("Recipe details": the activation quantizer selects
    between two scale factors per block).  Reading (the rule is not on the
    pages): each 16-value block is quantized twice with the same outer scale
    -- block maximum mapped to 6 (the plain rule) and to 4 -- and keeps the
    candidate with the smaller squared error (``block_sq_error_f32``); ties
    keep 6.  Returns (codes [R, C], scales [R, C/16], sg) and, when asked, the
    boolean [R, C/16] of blocks that took 4."""
    x = np.asarray(x, dtype=F32)
    R, C = x.shape
    if C % NVFP4_BLOCK:
        raise ValueError("C must be a multiple of 16")
    sg = outer_scale(x) if sg is None else F32(sg)
    xb = x.reshape(R * C // 16, 16)
    c6, s6 = _quantize_blocks(xb, sg, 6.0)
    c4, s4 = _quantize_blocks(xb, sg, 4.0)
    take4 = block_sq_error_f32(xb, c4, s4, sg) < block_sq_error_f32(xb, c6, s6, sg)
    codes = np.where(take4[:, None], c4, c6).reshape(R, C)
    scales = np.where(take4, s4, s6).reshape(R, C // 16)
    if return_choice:
        return codes, scales, sg, take4.reshape(R, C // 16)
    return codes, scales, sg


def quantize_col16(x, sg=None):
    """16x1 blocks (along columns): the backward-pass grouping that the page's
    Figure 2 compares with 1x16 ("Block-scaled backward passes")."""
    codes, scales, sg = quantize(np.asarray(x, dtype=F32).T, sg)
    return codes.T, scales.T, sg


def quantize_tile16x16(x, sg=None):
    """One E4M3 scale per 16x16 tile (NVIDIA's transpose-invariant weight
    scheme, Figure 3 of "Block-scaled backward passes").  Returns codes [R, C]
    and scales [R/16, C/16]."""
    x = np.asarray(x, dtype=F32)
    R, C = x.shape
    sg = outer_scale(x) if sg is None else F32(sg)
    tiles = x.reshape(R // 16, 16, C // 16, 16).transpose(0, 2, 1, 3).reshape(-1, 256)
    codes, scales = _quantize_blocks(tiles, sg)
    codes = codes.reshape(R // 16, C // 16, 16, 16).transpose(0, 2, 1, 3).reshape(R, C)
    return codes, scales.reshape(R // 16, C // 16), sg


def pack(codes) -> np.ndarray:
    """Pack 4-bit codes [R, C] into bytes [R, C/2]: low nibble = even element."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)


def unpack(packed) -> np.ndarray:
    """Inverse of ``pack``."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out


def dequantize_f32(codes, scales, sg) -> np.ndarray:
    """Dequantized values in fp32: fp32(fp32(e2m1 * e4m3) * sg).  The inner
    product is exact (at most 6 significant bits).  Used by the re-quantizer."""
    v = F.decode_e2m1_array(codes)
    s = F.decode_e4m3_array(np.repeat(np.asarray(scales, dtype=np.uint8), NVFP4_BLOCK, axis=-1))
    return ((v * s).astype(F32) * F32(sg)).astype(F32)


def dequantize_f64(codes, scales, sg) -> np.ndarray:
    """Exact dequantized values e2m1 * e4m3 * sg in float64 (GEMM references)."""
    v = F.decode_e2m1_array(codes)
    s = F.decode_e4m3_array(np.repeat(np.asarray(scales, dtype=np.uint8), NVFP4_BLOCK, axis=-1))
    return v * s * np.float64(F32(sg))


def dequantize_rows_f32(codes, scales, sg_rows) -> np.ndarray:
    """Per-token dequantization in fp32: fp32(fp32(e2m1 * e4m3) * sg_r)."""
    v = F.decode_e2m1_array(codes)
    s = F.decode_e4m3_array(np.repeat(np.asarray(scales, dtype=np.uint8), NVFP4_BLOCK, axis=-1))
    return ((v * s).astype(F32) * np.asarray(sg_rows, dtype=F32).reshape(-1, 1)).astype(F32)


def dequantize_rows_f64(codes, scales, sg_rows) -> np.ndarray:
    """Exact per-token dequantized values e2m1 * e4m3 * sg_r in float64."""
    v = F.decode_e2m1_array(codes)
    s = F.decode_e4m3_array(np.repeat(np.asarray(scales, dtype=np.uint8), NVFP4_BLOCK, axis=-1))
    return v * s * np.asarray(sg_rows, dtype=F32).astype(np.float64).reshape(-1, 1)


def dequantize_tile16x16_f64(codes, tile_scales, sg) -> np.ndarray:
    s = F.decode_e4m3_array(np.repeat(np.repeat(tile_scales, 16, axis=0), 16, axis=1))
    return F.decode_e2m1_array(codes) * s * np.float64(F32(sg))
