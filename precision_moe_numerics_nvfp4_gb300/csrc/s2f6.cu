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
#include "rht_s2f6_block.cuh"

namespace nvm {

// One block of 32 values per thread, moved with 32-byte loads and stores; the
// thread's next block is loaded before the current one is converted.
__global__ void __launch_bounds__(256) rht32_s2f6_quantize_kernel(const uint16_t *__restrict__ x, int64_t nblk,
                                                                  const RhtSigns sg, int8_t *__restrict__ codes,
                                                                  uint8_t *__restrict__ scales) {
  const int64_t threads = (int64_t)gridDim.x * blockDim.x;
  int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t next[16] = {};
  if (b < nblk) {
    ld_stream_v8(x + b * 32, reinterpret_cast<uint32_t(&)[8]>(next[0]));
    ld_stream_v8(x + b * 32 + 16, reinterpret_cast<uint32_t(&)[8]>(next[8]));
  }
  for (; b < nblk; b += threads) {
    uint32_t cur[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) cur[i] = next[i];
    const int64_t b1 = b + threads;
    if (b1 < nblk) {
      ld_stream_v8(x + b1 * 32, reinterpret_cast<uint32_t(&)[8]>(next[0]));
      ld_stream_v8(x + b1 * 32 + 16, reinterpret_cast<uint32_t(&)[8]>(next[8]));
    }
    uint32_t packed[8];
    const uint32_t sc = rht32_s2f6_block(cur, sg, packed);
    st_cs_v8(codes + b * 32, packed[0], packed[1], packed[2], packed[3], packed[4], packed[5], packed[6], packed[7]);
    scales[b] = (uint8_t)sc;
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
