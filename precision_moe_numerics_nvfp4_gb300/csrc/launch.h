// Host-side launchers shared between the translation units of libnvfp4moe.so.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "nvfp4moe.h"

namespace nvm {

int *status_ptr();  // device address of this device's status word (api.cu)

// largest iteration limit nvfp4moe_selftest_wait_timeout accepts
constexpr int64_t kMaxSelftestSpins = (int64_t)1 << 20;

// argument and shape checks of nvfp4_quantize (api.cu); NV_OK or NV_ERR_*
int quantize_check_args(const void *x, int64_t batch, int64_t rows, int64_t cols, const int32_t *group_offsets,
                        int32_t num_groups, const uint8_t *codes, const uint8_t *scales);
// the library's SR conversion on caller-given values and draws (misc.cu)
int launch_sr_e4m3x4(const float *x, const uint32_t *draws, int64_t n4, uint8_t *codes, cudaStream_t s);
// p[0 .. n) = v (one small kernel)
int launch_fill_f32(float *p, int64_t n, float v, cudaStream_t s);

int launch_amax(const uint16_t *x, int64_t batch, int64_t per_batch, float *partial, int nblk, float *sg_out,
                cudaStream_t s);
int launch_nvfp4_quant(const uint16_t *x, int64_t batch, int64_t rows, int64_t cols, const int32_t *groups, int E,
                       const float *sg, uint8_t *codes, uint8_t *scales, int *status, cudaStream_t s,
                       const float *sg_rows = nullptr, int four_six = 0);
// per-token outer scales sg_rows[r] = amax_r / 2688 (1 for a zero row); cols % 8 == 0
int launch_row_outer_scale(const uint16_t *x, int64_t rows, int64_t cols, float *sg_rows, cudaStream_t s);
int launch_mxfp8_rowwise(const uint16_t *x, int64_t rows, int64_t cols, const int32_t *groups, int E, int sr,
                         uint64_t seed, uint64_t off, uint8_t *codes, uint8_t *scales, int *status, cudaStream_t s);
int launch_mx_transpose_bf16(const uint16_t *x, int64_t rows, int64_t cols, const int32_t *groups, int E, int sr,
                             uint64_t seed, uint64_t off_t, uint64_t off_row, uint8_t *codes_t, uint8_t *scales_t,
                             uint8_t *codes_row, uint8_t *scales_row, int *status, cudaStream_t s);
int launch_requant(const uint8_t *codes, const uint8_t *scales, const float *sg, int64_t batch, int64_t rows,
                   int64_t cols, const int32_t *groups, int E, uint64_t seed, uint64_t off, uint8_t *out_codes,
                   uint8_t *out_scales, int *status, cudaStream_t s, const float *sg_rows = nullptr);
int launch_nvfp4_requant(const uint16_t *x, const float *sg, int64_t batch, int64_t rows, int64_t cols,
                         const int32_t *groups, int E, uint8_t *codes, uint8_t *scales, uint64_t seed, uint64_t off,
                         uint8_t *out_codes, uint8_t *out_scales, int *status, cudaStream_t s,
                         const float *sg_rows = nullptr, int four_six = 0, const int32_t *row_src = nullptr,
                         int64_t src_rows = 0);
// the re-quantization of gathered rows: routed row r is token row_src[r] of
// the NVFP4 token matrix (codes [src_rows][cols / 2], batched scale layout);
// writes the routed rows' NVFP4 codes and grouped scales and their
// transposed MXFP8 SR re-quantization
int launch_requant_gather(const uint8_t *tok_codes, const uint8_t *tok_scales, const float *sg,
                          const int32_t *row_src, int64_t src_rows, int64_t rows, int64_t cols,
                          const int32_t *groups, int E, uint8_t *codes, uint8_t *scales, uint64_t seed, uint64_t off,
                          uint8_t *out_codes, uint8_t *out_scales, int *status, cudaStream_t s);
// amax pass over the gathered rows x[row_src[r]] (r < rows) -> sg_out[0];
// row_amax: src_rows floats of scratch, used when src_rows <= rows
int launch_amax_gather(const uint16_t *x, const int32_t *row_src, int64_t src_rows, int64_t rows, int64_t cols,
                       float *partial, int nblk, float *row_amax, float *sg_out, int *status, cudaStream_t s);
int launch_outer_scale_from_amax(float *amax_in_sg_out, cudaStream_t s);
// per-row form: buf[r] = amax_r / 2688 (1 for zero) in place, r < n
int launch_row_outer_scale_from_amax(float *amax_in_sg_out, int64_t n, cudaStream_t s);
// RHT-32 + block-scaled S2F6 (s2f6.cu); n values, n % 32 == 0
int launch_rht32_s2f6_quantize(const uint16_t *x, int64_t n, uint32_t signs, int8_t *codes, uint8_t *scales,
                               cudaStream_t s);
int launch_s2f6_dequant_irht32(const int8_t *codes, const uint8_t *scales, int64_t n, uint32_t signs, void *y,
                               int y_fp32, cudaStream_t s);
int launch_swiglu_fwd(const uint16_t *y13, int64_t M, int64_t I, uint16_t *h, cudaStream_t s);
int launch_swiglu_bwd(const uint16_t *dh, const uint16_t *y13, int64_t M, int64_t I, uint16_t *dy13, cudaStream_t s);
int launch_wait_selftest(int64_t spins, int *status, cudaStream_t s);

// grouped GEMMs (gemm.cu)
// kGemmNvfp4FwdSwiglu: the w13 forward GEMM (N = 2I rows of gate over up per
// expert) with SwiGLU in the epilogue: y13 bf16, h bf16 and max |h|
enum GemmKind { kGemmNvfp4Fwd = 0, kGemmMxfp8Dx = 1, kGemmMxfp8Dw = 2, kGemmNvfp4FwdSwiglu = 3 };
struct GemmProblem {
  int kind;
  const uint8_t *a_codes, *a_scales, *b_codes, *b_scales;
  const float *a_sg, *b_sg;  // NVFP4 outer scales (fwd only)
  const int32_t *groups;
  int E;
  int64_t M_total, N, K;
  void *out;
  int out_fp32;
  void *h;                   // kGemmNvfp4FwdSwiglu: h [M_total][N / 2] bf16
  float *h_amax;             // kGemmNvfp4FwdSwiglu: max |h| accumulated (bits of a non-negative float)
  int a_sg_rows;             // 1: a_sg holds one outer scale per row of A (per token)
  int h_amax_rows;           // 1: h_amax holds one maximum per row of h
  // kGemmNvfp4Fwd with bf16 output: also RHT-32 + S2F6 of each row's bf16
  // values (codes int8 [M_total][N], scales u8 [M_total][N / 32]); out may
  // then be null (no bf16 output)
  int8_t *s2f6_codes;
  uint8_t *s2f6_scales;
  uint32_t rht_signs;
  // kGemmMxfp8Dx with bf16 output: the SwiGLU backward of the output dh with
  // y13 [M_total][2K] bf16; out is then dy13 [M_total][2K] bf16
  const uint16_t *swb_y13;
};
int launch_grouped_gemm(const GemmProblem &p, int *status, cudaStream_t s);
int set_gemm_variant(int v);  // 0 automatic, 1-3 forced (see nvfp4moe_set_gemm_kernel)
int set_gemm_wait_limit(int64_t spins);  // 0: default (see nvfp4moe_set_gemm_wait_limit)

}  // namespace nvm
