"""MXFP8 block quantization: 8-bit E4M3 elements, one E8M0 scale per 32
consecutive values, round-to-nearest or stochastic rounding.  Test
infrastructure only.

End-to-End 4-Bit Training, "Low-precision formats on Blackwell": the MX
formats scale blocks of 32 values with an E8M0 scale (8 exponent bits, no
sign, no mantissa).  "Re-quantization with stochastic rounding": weights and
activations are stochastically re-quantized to MXFP8 for the backward GEMMs.
Chinese translation, Figure 4 dataflow: the BF16 gradient is quantized to
MXFP8 with SR, once row-wise (for DGRAD) and once transposed (for WGRAD).

Conventions (the pages name neither the element type nor the scale rule):
  element type  E4M3 (largest finite 448, largest exponent 8)
  e             = floor(log2(bamax)), exact, from the exponent of bamax
  sexp          = clamp(e - 8, -127, 127), scale code = sexp + 127
  w             = fp32(v * 2^-sexp)
  code          = RN_E4M3(w) or SR_E4M3(w, R16), saturating at +-448
  bamax == 0   -> scale code 0x00 and signed-zero elements
Because the scale is a floor, |w| can reach [256, 512); values above 448
saturate, under SR too (the one biased case).
"""
from __future__ import annotations

import numpy as np

from . import formats as F

F32 = np.float32
MX_BLOCK = 32


def e8m0_scale(bamax):
    """(scale code uint8, sexp int64) for each block amax (float32 array)."""
    a = np.asarray(bamax, dtype=np.float64)
    _, ex = np.frexp(a)              # a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
    e = ex.astype(np.int64) - 1
    sexp = np.clip(e - 8, -127, 127)
    sexp = np.where(a == 0, -127, sexp)
    return (sexp + 127).astype(np.uint8), sexp


def quantize(v, mode: str = "rn", r16=None):
    """MXFP8 quantization of a float32 matrix [R, C] (C a multiple of 32),
    blocks along the row.  ``mode`` is "rn" or "sr"; SR needs ``r16`` [R, C]
    (16-bit random integers).  Returns (E4M3 codes [R, C], E8M0 codes
    [R, C/32])."""
    v = np.asarray(v, dtype=F32)
    R, C = v.shape
    if C % MX_BLOCK:
        raise ValueError("C must be a multiple of 32")
    vb = v.reshape(R, C // 32, 32)
    bamax = np.max(np.abs(vb), axis=2).astype(F32)
    scode, sexp = e8m0_scale(bamax)
    mult = np.ldexp(np.ones(sexp.shape, dtype=F32), (-sexp).astype(np.int32))  # exact 2^-sexp
    w = (vb * mult[:, :, None]).astype(F32)
    if mode == "rn":
        codes = F.rn_code(w, F.E4M3_TABLE)
    elif mode == "sr":
        if r16 is None:
            raise ValueError("SR needs random bits")
        codes = F.sr_code(w, F.E4M3_TABLE, np.asarray(r16).reshape(R, C // 32, 32))
    else:
        raise ValueError(mode)
    return codes.reshape(R, C).astype(np.uint8), scode.reshape(R, C // 32)


def dequantize_f64(codes, scales) -> np.ndarray:
    """Exact float64 values e4m3 * 2^(scale - 127)."""
    s = F.decode_e8m0_array(np.repeat(np.asarray(scales, dtype=np.uint8), MX_BLOCK, axis=-1))
    return F.decode_e4m3_array(codes) * s
