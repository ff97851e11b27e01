"""32-point random Hadamard transform (RHT) and block-scaled S2F6: the
quantizer of the combine direction.  Test infrastructure only.

End-to-End 4-Bit Training, "Quantized communications": before the combine
all-to-all the MoE output is rotated by a 32-dimensional random Hadamard
transform and quantized to block-scaled S2F6 -- a fixed-point format with two
signed integer bits and six fractional bits, values k/64 for k in
[-128, 127] (range -2 .. 127/64) -- with one scale factor per 32 values
(8.25 bits per value); the receiver dequantizes and inverts the transform,
which is orthogonal, preserves the energy and inverts exactly.

Readings (the pages state neither the sign source nor the scale rule):
  transform   y = H (d * x) / sqrt(32) on each block of 32 consecutive values
              of a row, H the Sylvester Hadamard matrix (entries +-1), d the
              random signs: bit i of a 32-bit mask negates element i
  inverse     x = d * (H y) / sqrt(32)   (H H = 32 I)
  scale       UE8M0 (the FP8 scale type of Blackwell's S2F6 conversions), as
              for MX formats: e = floor(log2(amax)), the largest S2F6 power of
              two is 2^0, so the scale is 2^e (clamped to [-127, 127]); the
              block maximum maps into [1, 2); amax == 0 -> code 0
  rounding    k = RN(v * 2^-e * 64) (ties to even), saturating to [-128, 127]

Two levels: `*_f64` is the definition (for the mathematical pins); the fp32
functions take the transform in single precision in a fixed order -- the
butterfly stages h = 1, 2, 4, 8, 16 with (a + b, a - b), then one multiply by
fp32(1/sqrt(32)) -- so that the S2F6 codes (integers decided by floating
point) are compared with a device computing in that precision and order.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
BLOCK = 32
S2F6_MIN, S2F6_MAX = -128, 127  # codes; value = code / 64
INV_SQRT32_F32 = F32(1.0 / np.sqrt(32.0))


def hadamard(n: int = BLOCK) -> np.ndarray:
    """Sylvester construction: H_1 = [1], H_2n = [[H, H], [H, -H]]."""
    h = np.ones((1, 1), dtype=np.int64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def signs_of(mask: int) -> np.ndarray:
    """+-1 per element of a block: bit i set -> element i negated."""
    return np.where((int(mask) >> np.arange(BLOCK)) & 1, -1.0, 1.0)


# ---- the definition (float64) ------------------------------------------------------
def rht_f64(x, mask: int) -> np.ndarray:
    """Blocks of 32 along the last axis: y = H (d x) / sqrt(32)."""
    x = np.asarray(x, dtype=np.float64)
    blocks = x.reshape(*x.shape[:-1], -1, BLOCK) * signs_of(mask)
    y = blocks @ hadamard().T / np.sqrt(BLOCK)
    return y.reshape(x.shape)


def irht_f64(y, mask: int) -> np.ndarray:
    y = np.asarray(y, dtype=np.float64)
    blocks = y.reshape(*y.shape[:-1], -1, BLOCK) @ hadamard().T / np.sqrt(BLOCK)
    return (blocks * signs_of(mask)).reshape(y.shape)


# ---- as computed in fp32 -------------------------------------------------------------
def _fwht_f32(blocks: np.ndarray) -> np.ndarray:
    """Unnormalized Walsh-Hadamard transform of the last axis (32) in float32,
    butterflies h = 1, 2, 4, 8, 16: (a, b) -> (a + b, a - b), a at index i with
    bit h clear, b at i + h."""
    v = np.array(blocks, dtype=F32, copy=True)
    h = 1
    while h < BLOCK:
        idx = np.arange(BLOCK)
        lo = idx[(idx & h) == 0]
        a, b = v[..., lo].copy(), v[..., lo + h].copy()
        v[..., lo] = a + b
        v[..., lo + h] = a - b
        h *= 2
    return v


def rht_f32(x, mask: int) -> np.ndarray:
    x = np.asarray(x, dtype=F32)
    blocks = x.reshape(*x.shape[:-1], -1, BLOCK) * signs_of(mask).astype(F32)
    return (_fwht_f32(blocks) * INV_SQRT32_F32).reshape(x.shape)


def irht_f32(y, mask: int) -> np.ndarray:
    y = np.asarray(y, dtype=F32)
    blocks = _fwht_f32(y.reshape(*y.shape[:-1], -1, BLOCK)) * INV_SQRT32_F32
    return (blocks * signs_of(mask).astype(F32)).reshape(y.shape)


# ---- block-scaled S2F6 ----------------------------------------------------------------
def s2f6_values() -> np.ndarray:
    """Every S2F6 value, code order -128 .. 127."""
    return np.arange(S2F6_MIN, S2F6_MAX + 1, dtype=np.float64) / 64.0


def e8m0_s2f6(amax):
    """(scale code uint8, e int64) per block amax: e = floor(log2 amax),
    clamped to [-127, 127]; amax == 0 -> e = -127 (code 0)."""
    a = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(a)
    e = np.clip(ex.astype(np.int64) - 1, -127, 127)
    e = np.where(a == 0, -127, e)
    return (e + 127).astype(np.uint8), e


def s2f6_quantize(v) -> tuple[np.ndarray, np.ndarray]:
    """float32 [..., C] (C % 32 == 0) -> (codes int8 [..., C], scales uint8
    [..., C/32]): per block, k = RN(v * 2^-e * 64), saturating."""
    v = np.asarray(v, dtype=F32)
    blocks = v.reshape(*v.shape[:-1], -1, BLOCK)
    amax = np.max(np.abs(blocks), axis=-1)
    code, e = e8m0_s2f6(amax)
    # v * 2^(6 - e) is exact (a power of two; values stay normal or exact subnormal)
    w = blocks.astype(np.float64) * np.ldexp(1.0, (6 - e)[..., None])
    k = np.clip(np.rint(w), S2F6_MIN, S2F6_MAX).astype(np.int8)  # rint: ties to even
    return k.reshape(v.shape), code


def s2f6_dequantize(codes, scales) -> np.ndarray:
    """k / 64 * 2^e as float32 (exact)."""
    k = np.asarray(codes, dtype=np.int8).astype(np.float64)
    blocks = k.reshape(*k.shape[:-1], -1, BLOCK)
    e = np.asarray(scales, dtype=np.int64) - 127
    return (blocks * np.ldexp(1.0, (e - 6)[..., None])).astype(F32).reshape(k.shape)


def rht_s2f6_quantize(x, mask: int):
    """bf16-valued float32 [rows, C] -> S2F6 codes and scales of rht_f32(x)."""
    return s2f6_quantize(rht_f32(x, mask))


def s2f6_dequantize_irht(codes, scales, mask: int) -> np.ndarray:
    """The receiver: dequantize, then the inverse transform (fp32)."""
    return irht_f32(s2f6_dequantize(codes, scales), mask)
