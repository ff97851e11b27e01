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

// Round-to-nearest-even to an integer, and back, for |v| < 2^22: adding
// 1.5 * 2^23 leaves the rounded integer in the low mantissa bits (the add
// rounds to nearest even); both directions are exact.
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
constexpr int kMagicBits = 0x4B400000;
__device__ __forceinline__ int rint_small(float v) { return __float_as_int(__fadd_rn(v, kMagic)) - kMagicBits; }
__device__ __forceinline__ float int_small_to_f(int k) { return __fsub_rn(__int_as_float(kMagicBits + k), kMagic); }

// 2^e as fp32 for e in [-127, 127] (2^-127 is subnormal)
__device__ __forceinline__ float pow2f_exact(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// One block of 32 values per thread, moved with 32-byte loads and stores; the
// thread's next block is loaded before the current one is converted.
__global__ void __launch_bounds__(256) rht32_s2f6_quantize_kernel(const uint16_t *__restrict__ x, int64_t nblk,
                                                                  uint32_t signs, int8_t *__restrict__ codes,
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
    uint32_t rw[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) rw[i] = next[i];
    const int64_t b1 = b + threads;
    if (b1 < nblk) {
      ld_stream_v8(x + b1 * 32, reinterpret_cast<uint32_t(&)[8]>(next[0]));
      ld_stream_v8(x + b1 * 32 + 16, reinterpret_cast<uint32_t(&)[8]>(next[8]));
    }
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j)  // bf16 -> fp32 with the random sign, one bit operation each
      v[j] = __uint_as_float(((j & 1) ? (rw[j >> 1] & 0xFFFF0000u) : (rw[j >> 1] << 16)) ^
                             (((signs >> j) & 1u) << 31));
    fwht32(v);
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      v[j] = __fmul_rn(v[j], c);
      m = fmaxf(m, fabsf(v[j]));
    }
    int e = -127;
    if (m > 0.0f) {
      e = floor_log2_nonzero(m);
      e = e < -127 ? -127 : (e > 127 ? 127 : e);
    }
    const float inv = pow2f_exact(-e);
    uint32_t packed[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) packed[i] = 0u;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      // y * 2^-e * 64: two exact power-of-two products (the first may only
      // lose bits of values that round to code 0 anyway)
      int k = rint_small(__fmul_rn(__fmul_rn(v[j], inv), 64.0f));
      k = k < -128 ? -128 : (k > 127 ? 127 : k);
      packed[j >> 2] |= ((uint32_t)k & 0xFFu) << (8 * (j & 3));
    }
    st_cs_v8(codes + b * 32, packed[0], packed[1], packed[2], packed[3], packed[4], packed[5], packed[6], packed[7]);
    scales[b] = (uint8_t)(e + 127);
  }
}

__global__ void __launch_bounds__(256) s2f6_dequant_irht32_kernel(const int8_t *__restrict__ codes,
                                                                  const uint8_t *__restrict__ scales, int64_t nblk,
                                                                  uint32_t signs, void *__restrict__ y,
                                                                  int y_fp32) {
  const int64_t threads = (int64_t)gridDim.x * blockDim.x;
  const float c = __uint_as_float(kInvSqrt32Bits);
  int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t next[8] = {};
  uint32_t next_sc = 0;
  if (b < nblk) {
    ld_stream_v8(codes + b * 32, next);
    next_sc = scales[b];
  }
  for (; b < nblk; b += threads) {
    uint32_t cw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) cw[i] = next[i];
    const float s = pow2f_exact((int)next_sc - 127);
    const int64_t b1 = b + threads;
    if (b1 < nblk) {
      ld_stream_v8(codes + b1 * 32, next);
      next_sc = scales[b1];
    }
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int k = (int)(int8_t)((cw[j >> 2] >> (8 * (j & 3))) & 0xFFu);
      v[j] = __fmul_rn(__fmul_rn(int_small_to_f(k), 0.015625f), s);  // k / 64 * 2^e, exact
    }
    fwht32(v);
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(__float_as_uint(__fmul_rn(v[j], c)) ^ (((signs >> j) & 1u) << 31));
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
      for (int i = 0; i < 16; ++i) o[i] = f32_to_bf16_bits(v[2 * i]) | (f32_to_bf16_bits(v[2 * i + 1]) << 16);
      uint16_t *dst = static_cast<uint16_t *>(y) + b * 32;
      st_cs_v8(dst, o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7]);
      st_cs_v8(dst + 16, o[8], o[9], o[10], o[11], o[12], o[13], o[14], o[15]);
    }
  }
}

static int grid_256(int64_t n) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
      sms = 148;
  }
  const int64_t ctas = (n / 32 + 255) / 256;  // one block of 32 values per thread
  const int64_t cap = (int64_t)sms * 4;      // grid-stride beyond four CTAs per SM
  return (int)(ctas < cap ? ctas : cap);
}

int launch_rht32_s2f6_quantize(const uint16_t *x, int64_t n, uint32_t signs, int8_t *codes, uint8_t *scales,
                               cudaStream_t s) {
  rht32_s2f6_quantize_kernel<<<grid_256(n), 256, 0, s>>>(x, n / 32, signs, codes, scales);
  return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

int launch_s2f6_dequant_irht32(const int8_t *codes, const uint8_t *scales, int64_t n, uint32_t signs, void *y,
                               int y_fp32, cudaStream_t s) {
  s2f6_dequant_irht32_kernel<<<grid_256(n), 256, 0, s>>>(codes, scales, n / 32, signs, y, y_fp32);
  return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

}  // namespace nvm
