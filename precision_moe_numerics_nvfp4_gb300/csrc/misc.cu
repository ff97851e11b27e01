// Elementwise SwiGLU between the two expert GEMMs (Figure 5 of the pages'
// Chinese translation: w13 GEMM -> quantize -> w2 GEMM), its backward, and
// the bounded-wait self-test.
#include "common.cuh"
#include "launch.h"

namespace nvm {


// h[m][j] = bf16(silu(gate) * up), gate = y13[m][j], up = y13[m][I + j]
__global__ void __launch_bounds__(256) swiglu_fwd_kernel(const uint16_t *__restrict__ y13, int64_t M, int64_t I,
                                                         uint16_t *__restrict__ h) {
  const int64_t per_row = I >> 3, n = M * per_row;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = t / per_row, j = (t - m * per_row) * 8;
    const uint4 g = ld_stream_v4(y13 + m * 2 * I + j);
    const uint4 u = ld_stream_v4(y13 + m * 2 * I + I + j);
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float g0 = bf16_lo(gw[k]), g1 = bf16_hi(gw[k]);
      const float h0 = swiglu_h(g0, bf16_lo(uw[k]));
      const float h1 = swiglu_h(g1, bf16_hi(uw[k]));
      o[k] = f32_to_bf16_bits(h0) | (f32_to_bf16_bits(h1) << 16);
    }
    *reinterpret_cast<uint4 *>(h + m * I + j) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// dgate = dh * up * s * (1 + gate * (1 - s)), dup = dh * gate * s, s = sigmoid(gate)
__global__ void __launch_bounds__(256) swiglu_bwd_kernel(const uint16_t *__restrict__ dh,
                                                         const uint16_t *__restrict__ y13, int64_t M, int64_t I,
                                                         uint16_t *__restrict__ dy13) {
  const int64_t per_row = I >> 3, n = M * per_row;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = t / per_row, j = (t - m * per_row) * 8;
    const uint4 g = ld_stream_v4(y13 + m * 2 * I + j);
    const uint4 u = ld_stream_v4(y13 + m * 2 * I + I + j);
    const uint4 d = ld_stream_v4(dh + m * I + j);
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w}, dw[4] = {d.x, d.y, d.z, d.w};
    uint32_t og[4], ou[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float gg[2] = {bf16_lo(gw[k]), bf16_hi(gw[k])};
      float uu[2] = {bf16_lo(uw[k]), bf16_hi(uw[k])};
      float dd[2] = {bf16_lo(dw[k]), bf16_hi(dw[k])};
      float dg0, dg1, du0, du1;
      swiglu_bwd_f32x2(dd[0], dd[1], gg[0], gg[1], uu[0], uu[1], dg0, dg1, du0, du1);
      og[k] = f32_to_bf16_bits(dg0) | (f32_to_bf16_bits(dg1) << 16);
      ou[k] = f32_to_bf16_bits(du0) | (f32_to_bf16_bits(du1) << 16);
    }
    *reinterpret_cast<uint4 *>(dy13 + m * 2 * I + j) = make_uint4(og[0], og[1], og[2], og[3]);
    *reinterpret_cast<uint4 *>(dy13 + m * 2 * I + I + j) = make_uint4(ou[0], ou[1], ou[2], ou[3]);
  }
}

// One CTA waits on an mbarrier that expects an arrival nobody makes; the
// bounded wait runs out and the kernel records NV_ERR_TIMEOUT.
__global__ void wait_selftest_kernel(int64_t spins, int *status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t a = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(a, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(a, 0, (uint64_t)spins)) record_error(status, NV_ERR_TIMEOUT);
}

__global__ void __launch_bounds__(256) fill_f32_kernel(float *__restrict__ p, int64_t n, float v) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    p[i] = v;
}

// Four fp32 values per thread through the library's stochastic rounding to
// E4M3 (cvt_e4m3x4_sr with the draw convention of the SR kernels: word i holds
// the draws U_a | U_b << 16 of values 4i .. 4i + 3)
__global__ void __launch_bounds__(256) sr_e4m3x4_kernel(const float4 *__restrict__ x,
                                                        const uint32_t *__restrict__ draws, int64_t n4,
                                                        uint32_t *__restrict__ out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = x[i];
    out[i] = cvt_e4m3x4_sr(v.x, v.y, v.z, v.w, ~draws[i]);
  }
}

static int grid_for(int64_t n) {
  int64_t g = (n + 255) / 256;
  if (g > 152 * 16) g = 152 * 16;
  return (int)(g < 1 ? 1 : g);
}

int launch_swiglu_fwd(const uint16_t *y13, int64_t M, int64_t I, uint16_t *h, cudaStream_t s) {
  swiglu_fwd_kernel<<<grid_for(M * I / 8), 256, 0, s>>>(y13, M, I, h);
  return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

int launch_swiglu_bwd(const uint16_t *dh, const uint16_t *y13, int64_t M, int64_t I, uint16_t *dy13, cudaStream_t s) {
  swiglu_bwd_kernel<<<grid_for(M * I / 8), 256, 0, s>>>(dh, y13, M, I, dy13);
  return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

int launch_sr_e4m3x4(const float *x, const uint32_t *draws, int64_t n4, uint8_t *codes, cudaStream_t s) {
  sr_e4m3x4_kernel<<<grid_for(n4), 256, 0, s>>>(reinterpret_cast<const float4 *>(x), draws, n4,
                                               reinterpret_cast<uint32_t *>(codes));
  return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

int launch_fill_f32(float *p, int64_t n, float v, cudaStream_t s) {
  if (n <= 0) return NV_OK;
  fill_f32_kernel<<<grid_for(n), 256, 0, s>>>(p, n, v);
  return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

int launch_wait_selftest(int64_t spins, int *status, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(spins, status);
  return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

}  // namespace nvm
