"""Number formats of the recipe, decoded from their bit fields, and rounding
onto their grids.  Test infrastructure only (see ``oracle/__init__.py``).

Sources
-------
End-to-End 4-Bit Training, "Low-precision formats on Blackwell":
  * FP4 (E2M1) holds +-{0, 0.5, 1, 1.5, 2, 3, 4, 6};
  * NVFP4 scales are E4M3 (one implicit sign bit, 4 exponent bits, 3 mantissa
    bits); MX scales are E8M0 (8 exponent bits, no sign, no mantissa).
Chinese translation of the same post, NVFP4 widget (the bit-field breakdown
of the worked example): the E4M3 scale 0|1101|100 reads
(-1)^0 x 2^(1101b - 0111b) x 1.100b = 96 (so the exponent bias is 7) and the
E2M1 value 0|11|1 reads (-1)^0 x 2^(11b - 01b) x 1.1b = 6 (bias 1).

Rounding conventions the pages leave open (stated once, shared with the
GPU library by contract, not by code):
  * RN = nearest grid value, ties to the code with an even least significant
    bit, saturating at the grid maximum, sign kept (so -0 exists);
  * SR = stochastic rounding between the two grid neighbours a <= |w| < b,
    rounding up iff R < floor(f * 2^16) with f = (|w| - a) / (b - a) and R a
    16-bit random integer; |w| >= max saturates.  "Re-quantization with
    stochastic rounding": round up or down with probability inversely
    proportional to the distance.
"""
from __future__ import annotations

import numpy as np

SR_BITS = 16  # random bits per element in stochastic rounding


# --------------------------------------------------------------------------
# Decoding from bit fields
# --------------------------------------------------------------------------
def e2m1_decode(code: int) -> float:
    """Value of a 4-bit E2M1 code: sign bit 3, exponent bits 2..1 (bias 1),
    mantissa bit 0.  Exponent field 0 is subnormal: 0.m x 2^(1-1)."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        mag = (m / 2.0) * 2.0 ** (1 - 1)
    else:
        mag = (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if s else mag


def e4m3_decode(code: int) -> float:
    """Value of an 8-bit E4M3 code: sign bit 7, exponent bits 6..3 (bias 7),
    mantissa bits 2..0.  Exponent field 0 is subnormal: 0.mmm x 2^(1-7).
    The all-ones pattern S.1111.111 is NaN and is never produced; the largest
    finite magnitude is 1.110b x 2^8 = 448."""
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 7
    if e == 0xF and m == 7:
        return float("nan")
    if e == 0:
        mag = (m / 8.0) * 2.0 ** (1 - 7)
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


def e8m0_decode(code: int) -> float:
    """Value of an E8M0 scale: 2^(code - 127); code 0xFF (NaN) never produced."""
    if code == 0xFF:
        return float("nan")
    return 2.0 ** (code - 127)


# Positive halves of the grids, as (magnitudes ascending, codes) tables.
E2M1_CODES = np.arange(0, 8, dtype=np.uint8)
E2M1_MAGS = np.array([e2m1_decode(int(c)) for c in E2M1_CODES], dtype=np.float64)
E4M3_CODES = np.arange(0, 0x7F, dtype=np.uint8)  # 0x00 .. 0x7E, NaN excluded
E4M3_MAGS = np.array([e4m3_decode(int(c)) for c in E4M3_CODES], dtype=np.float64)
E2M1_SIGN = np.uint8(0x8)
E4M3_SIGN = np.uint8(0x80)
E2M1_MAX = float(E2M1_MAGS[-1])   # 6
E4M3_MAX = float(E4M3_MAGS[-1])   # 448

E2M1_TABLE = (E2M1_MAGS, E2M1_CODES, E2M1_SIGN)
E4M3_TABLE = (E4M3_MAGS, E4M3_CODES, E4M3_SIGN)

_CHUNK = 1 << 16


def _signbit(v: np.ndarray) -> np.ndarray:
    return np.signbit(v)


def rn_code(v, table) -> np.ndarray:
    """Round-to-nearest code of each value: brute-force distance to every
    magnitude of the grid, ties to the even code, saturating (the nearest
    grid value to anything beyond the maximum is the maximum), sign kept.

    ``v`` is any float array (float32 values are exact in float64)."""
    mags, codes, sign = table
    v = np.asarray(v)
    flat = v.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    for lo in range(0, flat.size, _CHUNK):
        x = flat[lo:lo + _CHUNK].astype(np.float64)
        m = np.abs(x)
        d = np.abs(m[:, None] - mags[None, :])
        dmin = d.min(axis=1, keepdims=True)
        tie = d == dmin
        # among the nearest candidates prefer an even code; there are at most
        # two candidates and adjacent codes differ in their last bit
        even = (codes[None, :] & 1) == 0
        pick_even = tie & even
        has_even = pick_even.any(axis=1)
        idx = np.where(has_even, pick_even.argmax(axis=1), tie.argmax(axis=1))
        c = codes[idx]
        out[lo:lo + _CHUNK] = np.where(_signbit(x), c | sign, c)
    return out.reshape(v.shape)


def sr_code(v, table, r16) -> np.ndarray:
    """Stochastic-rounding code of each value given a 16-bit random integer
    per value.  With m = |v|: m >= max gives max; otherwise a = the largest
    grid magnitude <= m, b = the next one, f = (m - a)/(b - a), and the value
    rounds up to b iff R < floor(f * 2^16).  P(up) = floor(f 2^16) / 2^16, so
    E[SR(v)] = v exactly when f is a multiple of 2^-16 and otherwise the mean
    is below |v| by less than 2^-16 (b - a).  Sign kept."""
    mags, codes, sign = table
    v = np.asarray(v)
    r = np.asarray(r16, dtype=np.int64).reshape(-1)
    flat = v.reshape(-1)
    if r.size != flat.size:
        raise ValueError("one random integer per value")
    out = np.empty(flat.shape, dtype=np.uint8)
    top = mags.size - 1
    for lo in range(0, flat.size, _CHUNK):
        x = flat[lo:lo + _CHUNK].astype(np.float64)
        rr = r[lo:lo + _CHUNK]
        m = np.abs(x)
        sat = m >= mags[-1]
        # index of the largest grid magnitude <= m (brute force over the grid)
        le = m[:, None] >= mags[None, :]
        ia = np.where(sat, top, le.sum(axis=1) - 1)
        ib = np.minimum(ia + 1, top)
        a = mags[ia]
        b = mags[ib]
        with np.errstate(invalid="ignore", divide="ignore"):
            f = np.where(sat, 0.0, (m - a) / np.where(sat, 1.0, b - a))
        thresh = np.floor(f * float(1 << SR_BITS)).astype(np.int64)
        up = (~sat) & (rr < thresh)
        idx = np.where(up, ib, ia)
        c = codes[idx]
        out[lo:lo + _CHUNK] = np.where(_signbit(x), c | sign, c)
    return out.reshape(v.shape)


def decode_e2m1_array(codes) -> np.ndarray:
    """Float64 values of an array of 4-bit E2M1 codes."""
    lut = np.array([e2m1_decode(c) for c in range(16)], dtype=np.float64)
    return lut[np.asarray(codes, dtype=np.uint8) & 0xF]


def decode_e4m3_array(codes) -> np.ndarray:
    """Float64 values of an array of E4M3 codes."""
    lut = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return lut[np.asarray(codes, dtype=np.uint8)]


def decode_e8m0_array(codes) -> np.ndarray:
    """Float64 values of an array of E8M0 codes."""
    lut = np.array([e8m0_decode(c) for c in range(256)], dtype=np.float64)
    return lut[np.asarray(codes, dtype=np.uint8)]


def bf16_to_f32(bits_u16) -> np.ndarray:
    """Widen raw bf16 bit patterns (uint16) to float32 exactly."""
    b = np.asarray(bits_u16, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def f32_to_bf16_rne(x) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even) and return the
    raw uint16 patterns.  NaN is not expected."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) >> 16
    return u.astype(np.uint16)
