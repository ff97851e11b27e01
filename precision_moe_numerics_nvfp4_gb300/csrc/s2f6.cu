// 32-point random Hadamard transform + block-scaled S2F6, and the inverse
// ("End-to-End 4-Bit Training", "Quantized communications": the combine
// direction rotates each block of 32 values by a random Hadamard transform
// and quantizes to S2F6 -- two signed integer bits, six fractional bits,
// codes k/64 with k in [-128, 127] -- with one UE8M0 scale per 32 values).
//
// Layout: one block of 32 consecutive values per thread (a warp covers 32
// consecutive blocks).  The transform is the Walsh-Hadamard butterfly
// (a, b) -> (a + b, a - b) over the value index bits 0..4 in that order, in
// registers, then one multiply by fp32(1/sqrt(32)); the random signs (bit i of
// a 32-bit mask negates value i of every block) come first on the way in and
// last on the way out.  Scale: e = floor(log2(block max |y|)), the block
// maximum maps into [1, 2); code k = RN(y * 2^-e * 64) ties to even,
// saturating; an all-zero block gets scale code 0.  Memory bound: 2 bytes in,
// 1 + 1/32 bytes out per value (and the reverse).
#include "common.cuh"
#include "launch.h"

#include <cstring>

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

static RhtSigns make_signs(uint32_t signs) {
  RhtSigns r;
  const float c = [] { float f; uint32_t b = kInvSqrt32Bits; memcpy(&f, &b, 4); return f; }();
  for (int i = 0; i < 16; ++i) r.pair_mask[i] = ((signs >> (2 * i)) & 1u) << 15 | ((signs >> (2 * i + 1)) & 1u) << 31;
  for (int j = 0; j < 32; ++j) r.signed_c[j] = ((signs >> j) & 1u) ? -c : c;
  return r;
}

// One block of 32 values per thread, moved with 32-byte loads and stores; the
// thread's next block is loaded before the current one is converted.
//
// Arithmetic equal to the definition's fp32 order: y_j = fp32(t_j * c) with t
// the butterfly output.  Block max: max_j |y_j| = fp32(max_j |t_j| * c), since
// rounding is monotonic.  Codes: RN(y_j * 2^(6-e)); as the power-of-two
// product is exact, y_j * 2^(6-e) = fp32(t_j * (c * 2^(6-e))) whenever y_j is
// normal, and a subnormal y_j (|y_j| < 2^-126) gives |y_j| * 2^(6-e) < 1/4,
// code 0 either way, when e >= -118; below that the two products are taken
// in turn (c * 2^(6-e) would also leave the fp32 range).
__global__ void __launch_bounds__(256) rht32_s2f6_quantize_kernel(const uint16_t *__restrict__ x, int64_t nblk,
                                                                  const RhtSigns sg, int8_t *__restrict__ codes,
                                                                  uint8_t *__restrict__ scales) {
  const int64_t threads = (int64_t)gridDim.x * blockDim.x;
  const float c = __uint_as_float(kInvSqrt32Bits);
  int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t next[16] = {};
  if (b < nblk) {
    ld_stream_v8(x + b * 32, reinterpret_cast<uint32_t(&)[8]>(next[0]));
    ld_stream_v8(x + b * 32 + 16, reinterpret_cast<uint32_t(&)[8]>(next[8]));
  }
  for (; b < nblk; b += threads) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) {  // bf16 pair -> two fp32 with the random signs
      const uint32_t w = next[i] ^ sg.pair_mask[i];
      v[2 * i] = __uint_as_float(w << 16);
      v[2 * i + 1] = __uint_as_float(w & 0xFFFF0000u);
    }
    const int64_t b1 = b + threads;
    if (b1 < nblk) {
      ld_stream_v8(x + b1 * 32, reinterpret_cast<uint32_t(&)[8]>(next[0]));
      ld_stream_v8(x + b1 * 32 + 16, reinterpret_cast<uint32_t(&)[8]>(next[8]));
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
    uint32_t packed[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      packed[i] = __byte_perm(__byte_perm(q[4 * i], q[4 * i + 1], 0x0040), __byte_perm(q[4 * i + 2], q[4 * i + 3], 0x0040),
                              0x5410);
    st_cs_v8(codes + b * 32, packed[0], packed[1], packed[2], packed[3], packed[4], packed[5], packed[6], packed[7]);
    scales[b] = (uint8_t)(e + 127);
  }
}

// Inverse.  Code k -> k * 2^(e-6) exactly: with u = k + 128 (the code byte
// XOR 0x80), fp32 bits 0x4B400000 | u hold f = 1.5 * 2^23 + 128 + k, and
// fma(f, 2^(e-6), -(1.5 * 2^23 + 128) * 2^(e-6)) rounds k * 2^(e-6), which is
// representable, so it is exact; the constant fits fp32 for e <= 109 (above
// that the subtraction and the product are taken in turn).  The output signs
// ride on the multiply by +-c.
__global__ void __launch_bounds__(256) s2f6_dequant_irht32_kernel(const int8_t *__restrict__ codes,
                                                                  const uint8_t *__restrict__ scales, int64_t nblk,
                                                                  const RhtSigns sg, void *__restrict__ y,
                                                                  int y_fp32) {
  constexpr float kBias = 12583040.0f;  // 1.5 * 2^23 + 128
  const int64_t threads = (int64_t)gridDim.x * blockDim.x;
  int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // two blocks in flight per thread: 32 bytes each is too little to cover
  // the memory latency at this occupancy
  uint32_t n0[8] = {}, n1[8] = {};
  uint32_t sc0 = 0, sc1 = 0;
  if (b < nblk) {
    ld_stream_v8(codes + b * 32, n0);
    sc0 = scales[b];
  }
  if (b + threads < nblk) {
    ld_stream_v8(codes + (b + threads) * 32, n1);
    sc1 = scales[b + threads];
  }
  for (; b < nblk; b += threads) {
    float v[32];
    const int e = (int)sc0 - 127;
    const float p = pow2f_exact(e - 6);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t u = n0[i] ^ 0x80808080u;
#pragma unroll
      for (int j = 0; j < 4; ++j) v[4 * i + j] = __uint_as_float(__byte_perm(u, kMagicBits, 0x7650 | j));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) n0[i] = n1[i];
    sc0 = sc1;
    const int64_t b2 = b + 2 * threads;
    if (b2 < nblk) {
      ld_stream_v8(codes + b2 * 32, n1);
      sc1 = scales[b2];
    }
    if (e <= 109) {
      const float nb = -__fmul_rn(kBias, p);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __fmaf_rn(v[j], p, nb);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(__fsub_rn(v[j], kBias), p);
    }
    fwht32(v);
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(v[j], sg.signed_c[j]);
    if (y_fp32) {
      float *dst = static_cast<float *>(y) + b * 32;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        st_cs_v8(dst + 8 * i, __float_as_uint(v[8 * i]), __float_as_uint(v[8 * i + 1]), __float_as_uint(v[8 * i + 2]),
                 __float_as_uint(v[8 * i + 3]), __float_as_uint(v[8 * i + 4]), __float_as_uint(v[8 * i + 5]),
                 __float_as_uint(v[8 * i + 6]), __float_as_uint(v[8 * i + 7]));
    } else {
      uint32_t o[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i] = bf16x2_bits(v[2 * i], v[2 * i + 1]);
      uint16_t *dst = static_cast<uint16_t *>(y) + b * 32;
      st_cs_v8(dst, o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7]);
      st_cs_v8(dst + 16, o[8], o[9], o[10], o[11], o[12], o[13], o[14], o[15]);
    }
  }
}

// One thread per block of 32 values, grid-stride beyond one full wave (every
// resident CTA slot of every SM, from the kernel's occupancy)
template <typename Kernel>
static int grid_for(Kernel kernel, int64_t n, int *cached_wave) {
  if (*cached_wave == 0) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
      sms = 148;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0) != cudaSuccess || per_sm < 1)
      per_sm = 1;
    *cached_wave = sms * per_sm;
  }
  const int64_t ctas = (n / 32 + 255) / 256;
  return (int)(ctas < *cached_wave ? (ctas > 0 ? ctas : 1) : *cached_wave);
}

int launch_rht32_s2f6_quantize(const uint16_t *x, int64_t n, uint32_t signs, int8_t *codes, uint8_t *scales,
                               cudaStream_t s) {
  static int wave = 0;
  rht32_s2f6_quantize_kernel<<<grid_for(rht32_s2f6_quantize_kernel, n, &wave), 256, 0, s>>>(x, n / 32, make_signs(signs), codes, scales);
  return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

int launch_s2f6_dequant_irht32(const int8_t *codes, const uint8_t *scales, int64_t n, uint32_t signs, void *y,
                               int y_fp32, cudaStream_t s) {
  static int wave = 0;
  s2f6_dequant_irht32_kernel<<<grid_for(s2f6_dequant_irht32_kernel, n, &wave), 256, 0, s>>>(codes, scales, n / 32, make_signs(signs), y, y_fp32);
  return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

}  // namespace nvm
