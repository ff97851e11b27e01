// The C ABI of libnvfp4moe.so: argument checks, the per-device status word,
// and the launches of every step of the hot path.  See include/nvfp4moe.h for
// the contract of each entry point.
#include <algorithm>
#include <atomic>
#include <cstdio>

#include "common.cuh"
#include "launch.h"

namespace nvm {

// First error any kernel recorded on this device (0 = none).
static __device__ int g_status;

// Looked up once per device (with that device current) and cached; host
// threads that race on the first lookup store the same address, and the
// atomic makes that race well-defined.
int *status_ptr() {
  static std::atomic<int *> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  int *p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    void *a = nullptr;
    if (cudaGetSymbolAddress(&a, g_status) != cudaSuccess) return nullptr;
    p = static_cast<int *>(a);
    cache[dev].store(p, std::memory_order_release);
  }
  return p;
}

static bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool al4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
static bool al32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }  // GEMM outputs: 32-byte stores
static int64_t rup(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

static int amax_blocks(int64_t per_batch) {
  const int64_t n16 = per_batch / 8;
  int64_t nb = (n16 + 2047) / 2048;
  if (nb < 1) nb = 1;
  if (nb > 1216) nb = 1216;
  return (int)nb;
}

// The argument and shape checks of nvfp4_quantize (also run first by
// nvfp4_quantize_noalloc, so that both report the same error for the same
// bad call).  Empty shapes pass.
int quantize_check_args(const void *x, int64_t batch, int64_t rows, int64_t cols, const int32_t *group_offsets,
                        int32_t num_groups, const uint8_t *codes, const uint8_t *scales) {
  if (!x || !codes || !scales || batch < 1 || rows < 0 || cols < 0) return NV_ERR_ARG;
  if (cols % 16) return NV_ERR_SHAPE;
  if (group_offsets && (batch != 1 || num_groups < 1 || num_groups > kMaxGroups)) return NV_ERR_ARG;
  if (!al16(x) || !al16(codes) || !al16(scales) || !al16(group_offsets)) return NV_ERR_ALIGN;
  if (rows == 0 || cols == 0) return NV_OK;
  if (rows * cols / 16 >= (int64_t)1 << 31 || (group_offsets && rows >= (int64_t)1 << 30)) return NV_ERR_SHAPE;
  return NV_OK;
}

}  // namespace nvm

using namespace nvm;

extern "C" {

int64_t nvfp4moe_padded_cap(int64_t M_total, int64_t E) { return rup(M_total + 127 * E, 128); }

int64_t nvfp4moe_scale_bytes(int64_t padded_rows, int64_t kblocks) {
  return rup(padded_rows, 128) / 128 * ((kblocks + 3) / 4) * 512;
}

int64_t nvfp4moe_scale_offset(int64_t rp, int64_t c, int64_t kblocks) {
  return scale_offset(rp, c, (kblocks + 3) / 4);
}

size_t nvfp4moe_quantize_workspace_bytes(int64_t batch, int64_t rows, int64_t cols) {
  if (batch < 1 || rows < 0 || cols < 0) return 0;
  const int nb = amax_blocks(rows * cols);
  return (size_t)rup((batch * nb + batch) * 4, 256);
}

// the amax pass's partial maxima, then one float per token
// the amax pass's scratch, the token row maxima, then (src_rows <= rows) the
// tokens' NVFP4 codes and batched scales, each on a 256-byte boundary
static size_t gather_tok_codes_at(int64_t src_rows, int64_t rows, int64_t cols) {
  return nvfp4moe_quantize_workspace_bytes(1, rows, cols) + (size_t)rup(src_rows * 4, 256);
}
static size_t gather_tok_scales_at(int64_t src_rows, int64_t rows, int64_t cols) {
  return gather_tok_codes_at(src_rows, rows, cols) + (size_t)rup(std::max<int64_t>(src_rows * cols / 2, 1), 256);
}
size_t nvfp4moe_quantize_gather_workspace_bytes(int64_t src_rows, int64_t rows, int64_t cols) {
  if (src_rows < 0 || rows < 0 || cols < 0) return 0;
  if (src_rows > rows) return gather_tok_codes_at(src_rows, rows, cols);
  const int64_t tok_scales = nvfp4moe_scale_bytes(((src_rows + 127) / 128) * 128, cols / 16);
  return gather_tok_scales_at(src_rows, rows, cols) + (size_t)rup(std::max<int64_t>(tok_scales, 1), 256);
}

// codes, then the grouped scale buffer, then the outer scale, then the amax
// pass's workspace, each starting on a 256-byte boundary
size_t nvfp4moe_fwd_workspace_bytes(int64_t M_total, int64_t K, int64_t E) {
  if (M_total < 0 || K < 0 || E < 1) return 0;
  const size_t codes = (size_t)rup(M_total * K / 2, 256);
  const size_t scales = (size_t)rup(nvfp4moe_scale_bytes(nvfp4moe_padded_cap(M_total, E), K / 16), 256);
  return codes + scales + 256 + nvfp4moe_quantize_workspace_bytes(1, M_total, K);
}

const char *nvfp4moe_version(void) { return "nvfp4moe 0.1 (sm_103a)"; }

int nvfp4moe_set_gemm_kernel(int variant) { return nvm::set_gemm_variant(variant); }

int nvfp4moe_set_gemm_wait_limit(int64_t spins) { return nvm::set_gemm_wait_limit(spins); }

const char *nvfp4moe_status_string(int s) {
  switch (s) {
    case NV_OK: return "ok";
    case NV_ERR_ARG: return "invalid argument";
    case NV_ERR_ALIGN: return "pointer not 16-byte aligned";
    case NV_ERR_SHAPE: return "shape violates divisibility rules";
    case NV_ERR_OFFSETS: return "group offsets inconsistent";
    case NV_ERR_TIMEOUT: return "bounded wait ran out";
    case NV_ERR_CUDA: return "CUDA runtime error";
    case NV_ERR_UNSUPPORTED: return "unsupported";
    case NV_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int nvfp4moe_get_device_status(nv_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return NV_ERR_CUDA;
  int *p = status_ptr();
  if (!p) return NV_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return NV_ERR_CUDA;
  if (v != 0 && cudaMemset(p, 0, sizeof(int)) != cudaSuccess) return NV_ERR_CUDA;
  return v;
}

int nvfp4moe_selftest_wait_timeout(int64_t spins, nv_stream_t stream) {
  if (spins < 1 || spins > kMaxSelftestSpins) return NV_ERR_ARG;
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  return launch_wait_selftest(spins, st, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4moe_sr_e4m3x4(const float *x, const uint32_t *draws, int64_t n4, uint8_t *codes, nv_stream_t stream) {
  if (!x || !draws || !codes || n4 < 0) return NV_ERR_ARG;
  if (!al16(x) || !al4(draws) || !al4(codes)) return NV_ERR_ALIGN;
  if (n4 == 0) return NV_OK;
  return launch_sr_e4m3x4(x, draws, n4, codes, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_outer_scale(const void *x, int64_t batch, int64_t n, float *outer_scale_out, void *workspace,
                      size_t workspace_bytes, nv_stream_t stream) {
  if (!x || !outer_scale_out || batch < 1 || n < 0) return NV_ERR_ARG;
  if (n % 8) return NV_ERR_SHAPE;
  if (!al16(x) || !al4(outer_scale_out)) return NV_ERR_ALIGN;
  const size_t need = nvfp4moe_quantize_workspace_bytes(batch, 1, n);
  if (!workspace || workspace_bytes < need || !al16(workspace)) return NV_ERR_WORKSPACE;
  if (n == 0)  // an empty tensor: scale 1, written by a kernel (no host copy, so the call stays capturable)
    return launch_fill_f32(outer_scale_out, batch, 1.0f, reinterpret_cast<cudaStream_t>(stream));
  const int nb = amax_blocks(n);
  return launch_amax(static_cast<const uint16_t *>(x), batch, n, static_cast<float *>(workspace), nb,
                     outer_scale_out, reinterpret_cast<cudaStream_t>(stream));
}

static int quantize_impl(const void *x, int64_t batch, int64_t rows, int64_t cols, const int32_t *group_offsets,
                         int32_t num_groups, const float *outer_scale_in, float *outer_scale_out, uint8_t *codes,
                         uint8_t *scales, void *workspace, size_t workspace_bytes, nv_stream_t stream,
                         int four_six) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int chk = quantize_check_args(x, batch, rows, cols, group_offsets, num_groups, codes, scales);
  if (chk != NV_OK) return chk;
  if (rows == 0 || cols == 0) return NV_OK;
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  const float *sg = outer_scale_in;
  if (!outer_scale_in) {
    const size_t need = nvfp4moe_quantize_workspace_bytes(batch, rows, cols);
    if (!workspace || workspace_bytes < need || !al16(workspace)) return NV_ERR_WORKSPACE;
    const int nb = amax_blocks(rows * cols);
    float *partial = static_cast<float *>(workspace);
    float *dst = outer_scale_out ? outer_scale_out : partial + batch * nb;
    int r = launch_amax(static_cast<const uint16_t *>(x), batch, rows * cols, partial, nb, dst, s);
    if (r != NV_OK) return r;
    sg = dst;
  } else if (outer_scale_out && outer_scale_out != outer_scale_in) {
    if (cudaMemcpyAsync(outer_scale_out, outer_scale_in, batch * sizeof(float), cudaMemcpyDeviceToDevice, s) !=
        cudaSuccess)
      return NV_ERR_CUDA;
  }
  return launch_nvfp4_quant(static_cast<const uint16_t *>(x), batch, rows, cols, group_offsets, num_groups, sg, codes,
                            scales, st, s, nullptr, four_six);
}

int nvfp4_quantize(const void *x, int64_t batch, int64_t rows, int64_t cols, const int32_t *group_offsets,
                   int32_t num_groups, const float *outer_scale_in, float *outer_scale_out, uint8_t *codes,
                   uint8_t *scales, void *workspace, size_t workspace_bytes, nv_stream_t stream) {
  return quantize_impl(x, batch, rows, cols, group_offsets, num_groups, outer_scale_in, outer_scale_out, codes, scales,
                       workspace, workspace_bytes, stream, 0);
}

int nvfp4_quantize_four_over_six(const void *x, int64_t batch, int64_t rows, int64_t cols,
                                 const int32_t *group_offsets, int32_t num_groups, const float *outer_scale_in,
                                 float *outer_scale_out, uint8_t *codes, uint8_t *scales, void *workspace,
                                 size_t workspace_bytes, nv_stream_t stream) {
  return quantize_impl(x, batch, rows, cols, group_offsets, num_groups, outer_scale_in, outer_scale_out, codes, scales,
                       workspace, workspace_bytes, stream, 1);
}

static int quantize_requant_impl(const void *x, int64_t batch, int64_t rows, int64_t cols,
                                 const int32_t *group_offsets, int32_t num_groups, const float *outer_scale_in,
                                 float *outer_scale_out, uint8_t *codes, uint8_t *scales, void *workspace,
                                 size_t workspace_bytes, uint64_t seed, uint64_t counter_offset, uint8_t *out_codes,
                                 uint8_t *out_scales, nv_stream_t stream, int four_six) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!x || !codes || !scales || !out_codes || !out_scales || batch < 1 || rows < 0 || cols < 0) return NV_ERR_ARG;
  if (group_offsets && (batch != 1 || num_groups < 1 || num_groups > kMaxGroups)) return NV_ERR_ARG;
  if (cols % 128) return NV_ERR_SHAPE;
  if (!group_offsets && rows % 128) return NV_ERR_SHAPE;
  if (!al16(x) || !al16(codes) || !al16(scales) || !al16(out_codes) || !al16(out_scales) || !al16(group_offsets))
    return NV_ERR_ALIGN;
  if (rows == 0 || cols == 0) return NV_OK;
  if (rows >= (int64_t)1 << 30 || rows * cols / 16 >= (int64_t)1 << 31) return NV_ERR_SHAPE;
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  const float *sg = outer_scale_in;
  if (!outer_scale_in) {
    const size_t need = nvfp4moe_quantize_workspace_bytes(batch, rows, cols);
    if (!workspace || workspace_bytes < need || !al16(workspace)) return NV_ERR_WORKSPACE;
    const int nb = amax_blocks(rows * cols);
    float *partial = static_cast<float *>(workspace);
    float *dst = outer_scale_out ? outer_scale_out : partial + batch * nb;
    int r = launch_amax(static_cast<const uint16_t *>(x), batch, rows * cols, partial, nb, dst, s);
    if (r != NV_OK) return r;
    sg = dst;
  } else if (outer_scale_out && outer_scale_out != outer_scale_in) {
    if (cudaMemcpyAsync(outer_scale_out, outer_scale_in, batch * sizeof(float), cudaMemcpyDeviceToDevice, s) !=
        cudaSuccess)
      return NV_ERR_CUDA;
  }
  return launch_nvfp4_requant(static_cast<const uint16_t *>(x), sg, batch, rows, cols, group_offsets,
                              group_offsets ? num_groups : 0, codes, scales, seed, counter_offset, out_codes,
                              out_scales, st, s, nullptr, four_six);
}

int nvfp4_quantize_requant(const void *x, int64_t batch, int64_t rows, int64_t cols, const int32_t *group_offsets,
                           int32_t num_groups, const float *outer_scale_in, float *outer_scale_out, uint8_t *codes,
                           uint8_t *scales, void *workspace, size_t workspace_bytes, uint64_t seed,
                           uint64_t counter_offset, uint8_t *out_codes, uint8_t *out_scales, nv_stream_t stream) {
  return quantize_requant_impl(x, batch, rows, cols, group_offsets, num_groups, outer_scale_in, outer_scale_out, codes,
                               scales, workspace, workspace_bytes, seed, counter_offset, out_codes, out_scales, stream,
                               0);
}

int nvfp4_quantize_requant_four_over_six(const void *x, int64_t batch, int64_t rows, int64_t cols,
                                         const int32_t *group_offsets, int32_t num_groups,
                                         const float *outer_scale_in, float *outer_scale_out, uint8_t *codes,
                                         uint8_t *scales, void *workspace, size_t workspace_bytes, uint64_t seed,
                                         uint64_t counter_offset, uint8_t *out_codes, uint8_t *out_scales,
                                         nv_stream_t stream) {
  return quantize_requant_impl(x, batch, rows, cols, group_offsets, num_groups, outer_scale_in, outer_scale_out, codes,
                               scales, workspace, workspace_bytes, seed, counter_offset, out_codes, out_scales, stream,
                               1);
}

int nvfp4_quantize_requant_gather(const void *x, const int32_t *row_src, int64_t src_rows, int64_t rows,
                                  int64_t cols, const int32_t *group_offsets, int32_t num_groups,
                                  const float *outer_scale_in, float *outer_scale_out, uint8_t *codes,
                                  uint8_t *scales, void *workspace, size_t workspace_bytes, uint64_t seed,
                                  uint64_t counter_offset, uint8_t *out_codes, uint8_t *out_scales,
                                  nv_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!x || !row_src || !codes || !scales || !out_codes || !out_scales || !group_offsets || src_rows < 0 ||
      rows < 0 || cols < 0)
    return NV_ERR_ARG;
  if (num_groups < 1 || num_groups > kMaxGroups) return NV_ERR_ARG;
  if (cols % 128) return NV_ERR_SHAPE;
  if (!al16(x) || !al4(row_src) || !al16(codes) || !al16(scales) || !al16(out_codes) || !al16(out_scales) ||
      !al16(group_offsets))
    return NV_ERR_ALIGN;
  if (rows == 0 || cols == 0) return NV_OK;
  if (rows >= (int64_t)1 << 30 || src_rows >= (int64_t)1 << 31 || rows * cols / 16 >= (int64_t)1 << 31)
    return NV_ERR_SHAPE;
  // no more tokens than routed rows: the tokens are quantized once into the
  // workspace and the routed rows copied and re-quantized from their codes
  const bool tokens_once = src_rows <= rows;
  if ((!outer_scale_in || tokens_once) &&
      (!workspace || workspace_bytes < nvfp4moe_quantize_gather_workspace_bytes(src_rows, rows, cols) ||
       !al16(workspace)))
    return NV_ERR_WORKSPACE;
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  const float *sg = outer_scale_in;
  if (!outer_scale_in) {
    const int nb = amax_blocks(rows * cols);
    float *partial = static_cast<float *>(workspace);
    float *dst = outer_scale_out ? outer_scale_out : partial + nb;
    float *row_amax = partial + nvfp4moe_quantize_workspace_bytes(1, rows, cols) / 4;
    int r = launch_amax_gather(static_cast<const uint16_t *>(x), row_src, src_rows, rows, cols, partial, nb, row_amax,
                               dst, st, s);
    if (r != NV_OK) return r;
    sg = dst;
  } else if (outer_scale_out && outer_scale_out != outer_scale_in) {
    if (cudaMemcpyAsync(outer_scale_out, outer_scale_in, sizeof(float), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return NV_ERR_CUDA;
  }
  if (tokens_once) {
    // a routed row's NVFP4 codes and scales are its token's under the same
    // outer scale (the block rule sees one row at a time)
    uint8_t *tok_codes = static_cast<uint8_t *>(workspace) + gather_tok_codes_at(src_rows, rows, cols);
    uint8_t *tok_scales = static_cast<uint8_t *>(workspace) + gather_tok_scales_at(src_rows, rows, cols);
    int r = launch_nvfp4_quant(static_cast<const uint16_t *>(x), 1, src_rows, cols, nullptr, 0, sg, tok_codes,
                               tok_scales, st, s);
    if (r != NV_OK) return r;
    return launch_requant_gather(tok_codes, tok_scales, sg, row_src, src_rows, rows, cols, group_offsets, num_groups,
                                 codes, scales, seed, counter_offset, out_codes, out_scales, st, s);
  }
  return launch_nvfp4_requant(static_cast<const uint16_t *>(x), sg, 1, rows, cols, group_offsets, num_groups, codes,
                              scales, seed, counter_offset, out_codes, out_scales, st, s, nullptr, 0, row_src,
                              src_rows);
}

int rht32_s2f6_quantize(const void *x, int64_t rows, int64_t cols, uint32_t signs, int8_t *codes, uint8_t *scales,
                        nv_stream_t stream) {
  if (!x || !codes || !scales || rows < 0 || cols < 0) return NV_ERR_ARG;
  if (cols % 32) return NV_ERR_SHAPE;
  if (!al32(x) || !al32(codes)) return NV_ERR_ALIGN;
  if (rows == 0 || cols == 0) return NV_OK;
  return launch_rht32_s2f6_quantize(static_cast<const uint16_t *>(x), rows * cols, signs, codes, scales,
                                    reinterpret_cast<cudaStream_t>(stream));
}

int s2f6_dequantize_rht32_inverse(const int8_t *codes, const uint8_t *scales, int64_t rows, int64_t cols,
                                  uint32_t signs, void *y, int y_dtype, nv_stream_t stream) {
  if (!codes || !scales || !y || rows < 0 || cols < 0) return NV_ERR_ARG;
  if (y_dtype != NV_OUT_BF16 && y_dtype != NV_OUT_FP32) return NV_ERR_ARG;
  if (cols % 32) return NV_ERR_SHAPE;
  if (!al32(codes) || !al32(y)) return NV_ERR_ALIGN;
  if (rows == 0 || cols == 0) return NV_OK;
  return launch_s2f6_dequant_irht32(codes, scales, rows * cols, signs, y, y_dtype == NV_OUT_FP32,
                                    reinterpret_cast<cudaStream_t>(stream));
}

int mxfp8_quantize(const void *x, int64_t rows, int64_t cols, const int32_t *group_offsets, int32_t num_groups,
                   int mode, uint64_t seed, uint64_t counter_offset_row, uint64_t counter_offset_t,
                   uint8_t *codes_row, uint8_t *scales_row, uint8_t *codes_t, uint8_t *scales_t,
                   nv_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!x || rows < 0 || cols < 0 || (mode != NV_RN && mode != NV_SR)) return NV_ERR_ARG;
  if ((codes_row == nullptr) != (scales_row == nullptr) || (codes_t == nullptr) != (scales_t == nullptr))
    return NV_ERR_ARG;
  if (group_offsets && (num_groups < 1 || num_groups > kMaxGroups)) return NV_ERR_ARG;
  if (cols % 32) return NV_ERR_SHAPE;
  if (codes_t && cols % 128) return NV_ERR_SHAPE;
  if (!al16(x) || !al16(codes_row) || !al16(scales_row) || !al16(codes_t) || !al16(scales_t) || !al16(group_offsets))
    return NV_ERR_ALIGN;
  if (rows == 0 || cols == 0 || (!codes_row && !codes_t)) return NV_OK;
  if (rows >= (int64_t)1 << 30 || rows * cols >= (int64_t)1 << 40) return NV_ERR_SHAPE;
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  const int E = group_offsets ? num_groups : 0;
  const int sr = mode == NV_SR;
  if (codes_t)
    return launch_mx_transpose_bf16(static_cast<const uint16_t *>(x), rows, cols, group_offsets, E, sr, seed,
                                    counter_offset_t, counter_offset_row, codes_t, scales_t, codes_row, scales_row, st,
                                    s);
  return launch_mxfp8_rowwise(static_cast<const uint16_t *>(x), rows, cols, group_offsets, E, sr, seed,
                              counter_offset_row, codes_row, scales_row, st, s);
}

int dequant_transpose_requant_sr(const uint8_t *codes, const uint8_t *scales, const float *outer_scale, int64_t batch,
                                 int64_t rows, int64_t cols, const int32_t *group_offsets, int32_t num_groups,
                                 uint64_t seed, uint64_t counter_offset, uint8_t *out_codes, uint8_t *out_scales,
                                 nv_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!codes || !scales || !outer_scale || !out_codes || !out_scales || batch < 1 || rows < 0 || cols < 0)
    return NV_ERR_ARG;
  if (group_offsets && (batch != 1 || num_groups < 1 || num_groups > kMaxGroups)) return NV_ERR_ARG;
  if (cols % 128) return NV_ERR_SHAPE;
  if (!group_offsets && rows % 128) return NV_ERR_SHAPE;
  if (!al16(codes) || !al16(scales) || !al16(out_codes) || !al16(out_scales) || !al16(group_offsets))
    return NV_ERR_ALIGN;
  if (rows == 0 || cols == 0) return NV_OK;
  if (rows >= (int64_t)1 << 30) return NV_ERR_SHAPE;
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  return launch_requant(codes, scales, outer_scale, batch, rows, cols, group_offsets, group_offsets ? num_groups : 0,
                        seed, counter_offset, out_codes, out_scales, st, s);
}

// ---- per-token outer scales ------------------------------------------------------
// sg_rows_in NULL: the per-row amax pass writes sg_rows_out (required); else
// the given scales are used (and copied to sg_rows_out when that differs).
static int rows_scales(const void *x, int64_t rows, int64_t cols, const float *sg_rows_in, float *sg_rows_out,
                       const float **sg, cudaStream_t s) {
  if (!sg_rows_in) {
    if (!sg_rows_out) return NV_ERR_ARG;
    const int r = launch_row_outer_scale(static_cast<const uint16_t *>(x), rows, cols, sg_rows_out, s);
    if (r != NV_OK) return r;
    *sg = sg_rows_out;
    return NV_OK;
  }
  if (sg_rows_out && sg_rows_out != sg_rows_in &&
      cudaMemcpyAsync(sg_rows_out, sg_rows_in, rows * sizeof(float), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return NV_ERR_CUDA;
  *sg = sg_rows_in;
  return NV_OK;
}

int nvfp4_quantize_rows(const void *x, int64_t rows, int64_t cols, const int32_t *group_offsets, int32_t num_groups,
                        const float *sg_rows_in, float *sg_rows_out, uint8_t *codes, uint8_t *scales,
                        nv_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!x || !codes || !scales || rows < 0 || cols < 0) return NV_ERR_ARG;
  if (!sg_rows_in && !sg_rows_out) return NV_ERR_ARG;
  if (group_offsets && (num_groups < 1 || num_groups > kMaxGroups)) return NV_ERR_ARG;
  if (cols % 16) return NV_ERR_SHAPE;
  if (!al16(x) || !al16(codes) || !al16(scales) || !al16(group_offsets) || !al4(sg_rows_in) || !al4(sg_rows_out))
    return NV_ERR_ALIGN;
  if (rows == 0 || cols == 0) return NV_OK;
  if (rows * cols / 16 >= (int64_t)1 << 31 || rows >= (int64_t)1 << 30) return NV_ERR_SHAPE;
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  const float *sg = nullptr;
  int r = rows_scales(x, rows, cols, sg_rows_in, sg_rows_out, &sg, s);
  if (r != NV_OK) return r;
  return launch_nvfp4_quant(static_cast<const uint16_t *>(x), 1, rows, cols, group_offsets,
                            group_offsets ? num_groups : 0, sg, codes, scales, st, s, sg);
}

int nvfp4_quantize_requant_rows(const void *x, int64_t rows, int64_t cols, const int32_t *group_offsets,
                                int32_t num_groups, const float *sg_rows_in, float *sg_rows_out, uint8_t *codes,
                                uint8_t *scales, uint64_t seed, uint64_t counter_offset, uint8_t *out_codes,
                                uint8_t *out_scales, nv_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!x || !codes || !scales || !out_codes || !out_scales || rows < 0 || cols < 0) return NV_ERR_ARG;
  if (!sg_rows_in && !sg_rows_out) return NV_ERR_ARG;
  if (group_offsets && (num_groups < 1 || num_groups > kMaxGroups)) return NV_ERR_ARG;
  if (cols % 128) return NV_ERR_SHAPE;
  if (!group_offsets && rows % 128) return NV_ERR_SHAPE;
  if (!al16(x) || !al16(codes) || !al16(scales) || !al16(out_codes) || !al16(out_scales) || !al16(group_offsets) ||
      !al4(sg_rows_in) || !al4(sg_rows_out))
    return NV_ERR_ALIGN;
  if (rows == 0 || cols == 0) return NV_OK;
  if (rows >= (int64_t)1 << 30 || rows * cols / 16 >= (int64_t)1 << 31) return NV_ERR_SHAPE;
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  const float *sg = nullptr;
  int r = rows_scales(x, rows, cols, sg_rows_in, sg_rows_out, &sg, s);
  if (r != NV_OK) return r;
  return launch_nvfp4_requant(static_cast<const uint16_t *>(x), sg, 1, rows, cols, group_offsets,
                              group_offsets ? num_groups : 0, codes, scales, seed, counter_offset, out_codes,
                              out_scales, st, s, sg);
}

int dequant_transpose_requant_sr_rows(const uint8_t *codes, const uint8_t *scales, const float *sg_rows, int64_t rows,
                                      int64_t cols, const int32_t *group_offsets, int32_t num_groups, uint64_t seed,
                                      uint64_t counter_offset, uint8_t *out_codes, uint8_t *out_scales,
                                      nv_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!codes || !scales || !sg_rows || !out_codes || !out_scales || rows < 0 || cols < 0) return NV_ERR_ARG;
  if (group_offsets && (num_groups < 1 || num_groups > kMaxGroups)) return NV_ERR_ARG;
  if (cols % 128) return NV_ERR_SHAPE;
  if (!group_offsets && rows % 128) return NV_ERR_SHAPE;
  if (!al16(codes) || !al16(scales) || !al16(out_codes) || !al16(out_scales) || !al16(group_offsets) ||
      !al4(sg_rows))
    return NV_ERR_ALIGN;
  if (rows == 0 || cols == 0) return NV_OK;
  if (rows >= (int64_t)1 << 30) return NV_ERR_SHAPE;
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  return launch_requant(codes, scales, sg_rows, 1, rows, cols, group_offsets, group_offsets ? num_groups : 0, seed,
                        counter_offset, out_codes, out_scales, st, s, sg_rows);
}

static int gemm_common_checks(const int32_t *go, int32_t E, int64_t M_total, int64_t N, int64_t K) {
  if (!go || E < 1 || E > kMaxGroups || M_total < 0 || N <= 0 || K <= 0) return NV_ERR_ARG;
  if (!al16(go)) return NV_ERR_ALIGN;
  if (M_total >= (int64_t)1 << 30) return NV_ERR_SHAPE;
  return NV_OK;
}

int grouped_gemm_nvfp4_fwd(const void *x_bf16, const float *x_outer_scale, const uint8_t *x_codes,
                           const uint8_t *x_scales, const uint8_t *w_codes, const uint8_t *w_scales,
                           const float *w_outer_scale, const int32_t *group_offsets, int32_t E, int64_t M_total,
                           int64_t N, int64_t K, void *y, int y_dtype, void *workspace, size_t workspace_bytes,
                           nv_stream_t stream) {
  int r = gemm_common_checks(group_offsets, E, M_total, N, K);
  if (r != NV_OK) return r;
  if (!w_codes || !w_scales || !w_outer_scale || !y) return NV_ERR_ARG;
  if (!x_bf16 && (!x_outer_scale || !x_codes || !x_scales)) return NV_ERR_ARG;
  if (y_dtype != NV_OUT_BF16 && y_dtype != NV_OUT_FP32) return NV_ERR_ARG;
  if (N % 128 || K % 256) return NV_ERR_SHAPE;
  if (!al16(w_codes) || !al16(w_scales) || !al32(y)) return NV_ERR_ALIGN;
  if (!x_bf16 && (!al16(x_codes) || !al16(x_scales))) return NV_ERR_ALIGN;
  if (x_bf16) {
    // the activations arrive in bf16: quantize them (nvfp4_quantize, grouped
    // layout, outer scale given or computed) into the workspace, then the GEMM
    if (!al16(x_bf16)) return NV_ERR_ALIGN;
    const size_t need = nvfp4moe_fwd_workspace_bytes(M_total, K, E);
    if (!workspace || workspace_bytes < need || !al16(workspace)) return NV_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t cb = (size_t)rup(M_total * K / 2, 256);
    const size_t sb = (size_t)rup(nvfp4moe_scale_bytes(nvfp4moe_padded_cap(M_total, E), K / 16), 256);
    uint8_t *codes = ws, *scales = ws + cb;
    float *sg = reinterpret_cast<float *>(ws + cb + sb);
    void *qws = ws + cb + sb + 256;
    r = quantize_impl(x_bf16, 1, M_total, K, group_offsets, E, x_outer_scale, sg, codes, scales, qws,
                      workspace_bytes - (cb + sb + 256), stream, 0);
    if (r != NV_OK) return r;
    x_codes = codes;
    x_scales = scales;
    x_outer_scale = sg;
  }
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  GemmProblem p = {kGemmNvfp4Fwd, x_codes, x_scales, w_codes, w_scales, x_outer_scale, w_outer_scale,
                   group_offsets, E, M_total, N, K, y, y_dtype == NV_OUT_FP32};
  return launch_grouped_gemm(p, st, reinterpret_cast<cudaStream_t>(stream));
}

int grouped_gemm_nvfp4_fwd_swiglu(const float *x_outer_scale, const uint8_t *x_codes, const uint8_t *x_scales,
                                  const uint8_t *w_codes, const uint8_t *w_scales, const float *w_outer_scale,
                                  const int32_t *group_offsets, int32_t E, int64_t M_total, int64_t I, int64_t K,
                                  void *y13, void *h, float *h_outer_scale, nv_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (I <= 0) return NV_ERR_ARG;
  int r = gemm_common_checks(group_offsets, E, M_total, 2 * I, K);
  if (r != NV_OK) return r;
  if (!x_outer_scale || !x_codes || !x_scales || !w_codes || !w_scales || !w_outer_scale || !y13 || !h ||
      !h_outer_scale)
    return NV_ERR_ARG;
  if (I % 128 || K % 256) return NV_ERR_SHAPE;
  if (!al16(x_codes) || !al16(x_scales) || !al16(w_codes) || !al16(w_scales) || !al32(y13) || !al32(h) ||
      !al16(h_outer_scale))
    return NV_ERR_ALIGN;
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  if (cudaMemsetAsync(h_outer_scale, 0, sizeof(float), s) != cudaSuccess) return NV_ERR_CUDA;
  if (M_total > 0) {
    GemmProblem p = {kGemmNvfp4FwdSwiglu, x_codes, x_scales, w_codes, w_scales, x_outer_scale, w_outer_scale,
                     group_offsets, E, M_total, 2 * I, K, y13, 0, h, h_outer_scale};
    r = launch_grouped_gemm(p, st, s);
    if (r != NV_OK) return r;
  }
  return launch_outer_scale_from_amax(h_outer_scale, s);
}

int grouped_gemm_nvfp4_fwd_rht_s2f6(const float *x_outer_scale, const uint8_t *x_codes, const uint8_t *x_scales,
                                    const uint8_t *w_codes, const uint8_t *w_scales, const float *w_outer_scale,
                                    const int32_t *group_offsets, int32_t E, int64_t M_total, int64_t N, int64_t K,
                                    uint32_t signs, void *y, int8_t *codes, uint8_t *scales, nv_stream_t stream) {
  int r = gemm_common_checks(group_offsets, E, M_total, N, K);
  if (r != NV_OK) return r;
  if (!x_outer_scale || !x_codes || !x_scales || !w_codes || !w_scales || !w_outer_scale || !codes || !scales)
    return NV_ERR_ARG;
  if (N % 128 || K % 256) return NV_ERR_SHAPE;
  if (!al16(x_codes) || !al16(x_scales) || !al16(w_codes) || !al16(w_scales) || !al32(y) || !al32(codes))
    return NV_ERR_ALIGN;
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  GemmProblem p = {kGemmNvfp4Fwd, x_codes, x_scales, w_codes, w_scales, x_outer_scale, w_outer_scale,
                   group_offsets, E, M_total, N, K, y, 0, nullptr, nullptr, 0, 0, codes, scales, signs};
  return launch_grouped_gemm(p, st, reinterpret_cast<cudaStream_t>(stream));
}

int grouped_gemm_nvfp4_fwd_rows(const float *x_sg_rows, const uint8_t *x_codes, const uint8_t *x_scales,
                                const uint8_t *w_codes, const uint8_t *w_scales, const float *w_outer_scale,
                                const int32_t *group_offsets, int32_t E, int64_t M_total, int64_t N, int64_t K,
                                void *y, int y_dtype, nv_stream_t stream) {
  int r = gemm_common_checks(group_offsets, E, M_total, N, K);
  if (r != NV_OK) return r;
  if (!x_sg_rows || !x_codes || !x_scales || !w_codes || !w_scales || !w_outer_scale || !y) return NV_ERR_ARG;
  if (y_dtype != NV_OUT_BF16 && y_dtype != NV_OUT_FP32) return NV_ERR_ARG;
  if (N % 128 || K % 256) return NV_ERR_SHAPE;
  if (!al16(x_codes) || !al16(x_scales) || !al16(w_codes) || !al16(w_scales) || !al32(y) || !al4(x_sg_rows))
    return NV_ERR_ALIGN;
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  GemmProblem p = {kGemmNvfp4Fwd, x_codes, x_scales, w_codes, w_scales, x_sg_rows, w_outer_scale,
                   group_offsets, E, M_total, N, K, y, y_dtype == NV_OUT_FP32, nullptr, nullptr, 1, 0};
  return launch_grouped_gemm(p, st, reinterpret_cast<cudaStream_t>(stream));
}

int grouped_gemm_nvfp4_fwd_swiglu_rows(const float *x_sg_rows, const uint8_t *x_codes, const uint8_t *x_scales,
                                       const uint8_t *w_codes, const uint8_t *w_scales, const float *w_outer_scale,
                                       const int32_t *group_offsets, int32_t E, int64_t M_total, int64_t I, int64_t K,
                                       void *y13, void *h, float *h_sg_rows, nv_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (I <= 0) return NV_ERR_ARG;
  int r = gemm_common_checks(group_offsets, E, M_total, 2 * I, K);
  if (r != NV_OK) return r;
  if (!x_sg_rows || !x_codes || !x_scales || !w_codes || !w_scales || !w_outer_scale || !y13 || !h || !h_sg_rows)
    return NV_ERR_ARG;
  if (I % 128 || K % 256) return NV_ERR_SHAPE;
  if (!al16(x_codes) || !al16(x_scales) || !al16(w_codes) || !al16(w_scales) || !al32(y13) || !al32(h) ||
      !al4(x_sg_rows) || !al4(h_sg_rows))
    return NV_ERR_ALIGN;
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  if (M_total == 0) return NV_OK;
  if (cudaMemsetAsync(h_sg_rows, 0, M_total * sizeof(float), s) != cudaSuccess) return NV_ERR_CUDA;
  GemmProblem p = {kGemmNvfp4FwdSwiglu, x_codes, x_scales, w_codes, w_scales, x_sg_rows, w_outer_scale,
                   group_offsets, E, M_total, 2 * I, K, y13, 0, h, h_sg_rows, 1, 1};
  r = launch_grouped_gemm(p, st, s);
  if (r != NV_OK) return r;
  return launch_row_outer_scale_from_amax(h_sg_rows, M_total, s);
}

int grouped_gemm_mxfp8_dx(const uint8_t *g_codes, const uint8_t *g_scales, const uint8_t *wt_codes,
                          const uint8_t *wt_scales, const int32_t *group_offsets, int32_t E, int64_t M_total,
                          int64_t N, int64_t K, void *dx, int dx_dtype, void *workspace, size_t workspace_bytes,
                          nv_stream_t stream) {
  (void)workspace; (void)workspace_bytes;
  int r = gemm_common_checks(group_offsets, E, M_total, N, K);
  if (r != NV_OK) return r;
  if (!g_codes || !g_scales || !wt_codes || !wt_scales || !dx) return NV_ERR_ARG;
  if (dx_dtype != NV_OUT_BF16 && dx_dtype != NV_OUT_FP32) return NV_ERR_ARG;
  if (N % 128 || K % 128) return NV_ERR_SHAPE;
  if (!al16(g_codes) || !al16(g_scales) || !al16(wt_codes) || !al16(wt_scales) || !al32(dx)) return NV_ERR_ALIGN;
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  GemmProblem p = {kGemmMxfp8Dx, g_codes, g_scales, wt_codes, wt_scales, nullptr, nullptr,
                   group_offsets, E, M_total, N, K, dx, dx_dtype == NV_OUT_FP32};
  return launch_grouped_gemm(p, st, reinterpret_cast<cudaStream_t>(stream));
}

int grouped_gemm_mxfp8_dx_swiglu_bwd(const uint8_t *g_codes, const uint8_t *g_scales, const uint8_t *wt_codes,
                                     const uint8_t *wt_scales, const int32_t *group_offsets, int32_t E,
                                     int64_t M_total, int64_t N, int64_t I, const void *y13, void *dy13,
                                     nv_stream_t stream) {
  int r = gemm_common_checks(group_offsets, E, M_total, N, I);
  if (r != NV_OK) return r;
  if (!g_codes || !g_scales || !wt_codes || !wt_scales || !y13 || !dy13) return NV_ERR_ARG;
  if (N % 128 || I % 128) return NV_ERR_SHAPE;
  if (!al16(g_codes) || !al16(g_scales) || !al16(wt_codes) || !al16(wt_scales) || !al32(y13) || !al32(dy13))
    return NV_ERR_ALIGN;
  const uintptr_t yb = reinterpret_cast<uintptr_t>(y13), db = reinterpret_cast<uintptr_t>(dy13);
  const uintptr_t bytes = (uintptr_t)(M_total * 2 * I * 2);
  if (yb < db + bytes && db < yb + bytes) return NV_ERR_ARG;  // y13 and dy13 overlap
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  GemmProblem p = {kGemmMxfp8Dx, g_codes, g_scales, wt_codes, wt_scales, nullptr, nullptr,
                   group_offsets, E, M_total, N, I, dy13, 0};
  p.swb_y13 = static_cast<const uint16_t *>(y13);
  return launch_grouped_gemm(p, st, reinterpret_cast<cudaStream_t>(stream));
}

int grouped_gemm_mxfp8_dw(const uint8_t *gt_codes, const uint8_t *gt_scales, const uint8_t *xt_codes,
                          const uint8_t *xt_scales, const int32_t *group_offsets, int32_t E, int64_t M_total,
                          int64_t N, int64_t K, float *dw, void *workspace, size_t workspace_bytes,
                          nv_stream_t stream) {
  (void)workspace; (void)workspace_bytes;
  int r = gemm_common_checks(group_offsets, E, M_total, N, K);
  if (r != NV_OK) return r;
  if (!gt_codes || !gt_scales || !xt_codes || !xt_scales || !dw) return NV_ERR_ARG;
  if (N % 128 || K % 128) return NV_ERR_SHAPE;
  if (!al16(gt_codes) || !al16(gt_scales) || !al16(xt_codes) || !al16(xt_scales) || !al32(dw)) return NV_ERR_ALIGN;
  int *st = status_ptr();
  if (!st) return NV_ERR_CUDA;
  GemmProblem p = {kGemmMxfp8Dw, gt_codes, gt_scales, xt_codes, xt_scales, nullptr, nullptr,
                   group_offsets, E, M_total, N, K, dw, 1};
  return launch_grouped_gemm(p, st, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4moe_swiglu_fwd(const void *y13, int64_t M, int64_t I, void *h, nv_stream_t stream) {
  if (!y13 || !h || M < 0 || I <= 0) return NV_ERR_ARG;
  if (I % 8) return NV_ERR_SHAPE;
  if (!al16(y13) || !al16(h)) return NV_ERR_ALIGN;
  if (M == 0) return NV_OK;
  return launch_swiglu_fwd(static_cast<const uint16_t *>(y13), M, I, static_cast<uint16_t *>(h),
                           reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4moe_swiglu_bwd(const void *dh, const void *y13, int64_t M, int64_t I, void *dy13, nv_stream_t stream) {
  if (!dh || !y13 || !dy13 || M < 0 || I <= 0) return NV_ERR_ARG;
  if (I % 8) return NV_ERR_SHAPE;
  if (!al16(dh) || !al16(y13) || !al16(dy13)) return NV_ERR_ALIGN;
  if (M == 0) return NV_OK;
  return launch_swiglu_bwd(static_cast<const uint16_t *>(dh), static_cast<const uint16_t *>(y13), M, I,
                           static_cast<uint16_t *>(dy13), reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
