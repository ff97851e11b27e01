// RHT-32 + block-scaled S2F6 arithmetic of one block of 32 values, shared by
// the standalone quantizer (s2f6.cu) and the forward GEMM's epilogue
// (gemm.cu), so that both produce the same codes bit for bit.
// "End-to-End 4-Bit Training", "Quantized communications": each block of 32
// values is rotated by a random Hadamard transform and quantized to S2F6
// (codes k/64, k in [-128, 127]) with one UE8M0 scale per block.
#pragma once
#include <cstdint>
#include <cstring>

#include "common.cuh"

namespace nvm {

constexpr uint32_t kInvSqrt32Bits = 0x3e3504f3u;  // fp32 nearest to 1/sqrt(32)

// the unnormalized Walsh-Hadamard butterfly of one block in registers:
// stages h = 1, 2, 4, 8, 16, (a, b) -> (a + b, a - b)
__device__ __forceinline__ void fwht32(float (&v)[32]) {
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if ((j & h) == 0) {
        const float a = v[j], b = v[j + h];
        v[j] = a + b;
        v[j + h] = a - b;
      }
    }
  }
}

// The magic number 1.5 * 2^23: for |w| < 2^22 the sum w + 1.5 * 2^23 lies in
// [2^23, 2^24), where fp32 steps by 1, so the add rounds w to the nearest
// integer (ties to even) and leaves it in the low mantissa bits: bits(sum) =
// 0x4B400000 + RN(w), monotonic in w, low byte = RN(w) mod 256.
constexpr float kMagic = 12582912.0f;
constexpr uint32_t kMagicBits = 0x4B400000u;

// 2^e as fp32 for e in [-149, 127] (subnormal below -126), exact
__device__ __forceinline__ float pow2f_exact(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(1u << (e + 149));
}

// Per-mask constants, passed by value so that they sit in the constant bank
// and unrolled code reads them as instruction operands (no registers):
// pair_mask[i] flips the sign bits of values 2i (bit 15) and 2i + 1 (bit 31)
// of a bf16 pair, signed_c[j] = +-fp32(1/sqrt(32)) carries d[j].
struct RhtSigns {
  uint32_t pair_mask[16];
  float signed_c[32];
};

inline RhtSigns make_signs(uint32_t signs) {
  RhtSigns r;
  const float c = [] { float f; uint32_t b = kInvSqrt32Bits; memcpy(&f, &b, 4); return f; }();
  for (int i = 0; i < 16; ++i) r.pair_mask[i] = ((signs >> (2 * i)) & 1u) << 15 | ((signs >> (2 * i + 1)) & 1u) << 31;
  for (int j = 0; j < 32; ++j) r.signed_c[j] = ((signs >> j) & 1u) ? -c : c;
  return r;
}

// One block: 16 words of bf16 pairs (value 2i in the low half of word i) ->
// 32 S2F6 codes (byte j of packed[j / 4] is code j) and the scale code.
//
// Arithmetic equal to the definition's fp32 order: y_j = fp32(t_j * c) with t
// the butterfly output.  Block max: max_j |y_j| = fp32(max_j |t_j| * c), since
// rounding is monotonic.  Codes: RN(y_j * 2^(6-e)); as the power-of-two
// product is exact, y_j * 2^(6-e) = fp32(t_j * (c * 2^(6-e))) whenever y_j is
// normal, and a subnormal y_j (|y_j| < 2^-126) gives |y_j| * 2^(6-e) < 1/4,
// code 0 either way, when e >= -118; below that the two products are taken
// in turn (c * 2^(6-e) would also leave the fp32 range).
__device__ __forceinline__ uint32_t rht32_s2f6_block(const uint32_t (&w16)[16], const RhtSigns &sg,
                                                     uint32_t (&packed)[8]) {
  const float c = __uint_as_float(kInvSqrt32Bits);
  float v[32];
#pragma unroll
  for (int i = 0; i < 16; ++i) {  // bf16 pair -> two fp32 with the random signs
    const uint32_t w = w16[i] ^ sg.pair_mask[i];
    v[2 * i] = __uint_as_float(w << 16);
    v[2 * i + 1] = __uint_as_float(w & 0xFFFF0000u);
  }
  fwht32(v);
  float tm = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) tm = fmaxf(tm, fabsf(v[j]));
  const float m = __fmul_rn(tm, c);
  int e = -127;
  if (m > 0.0f) {
    e = floor_log2_nonzero(m);
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
  }
  uint32_t q[32];
  if (e >= -118) {
    const float qs = __fmul_rn(c, pow2f_exact(6 - e));
#pragma unroll
    for (int j = 0; j < 32; ++j) q[j] = __float_as_uint(__fadd_rn(__fmul_rn(v[j], qs), kMagic));
  } else {
    const float up = pow2f_exact(6 - e - 64);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      q[j] = __float_as_uint(__fadd_rn(__fmul_rn(__fmul_rn(__fmul_rn(v[j], c), 18446744073709551616.0f), up), kMagic));
  }
  // |w| < 128 by the choice of e, so RN gives [-128, 128]: saturate the top
#pragma unroll
  for (int j = 0; j < 32; ++j) q[j] = min(q[j], kMagicBits + 127u);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    packed[i] = __byte_perm(__byte_perm(q[4 * i], q[4 * i + 1], 0x0040), __byte_perm(q[4 * i + 2], q[4 * i + 3], 0x0040),
                            0x5410);
  return (uint32_t)(e + 127);
}

}  // namespace nvm
