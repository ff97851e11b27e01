// Quantization kernels of libnvfp4moe.so (HBM-bound):
//   amax_partial / outer_scale_finalize   per-tensor amax -> FP32 outer scale sg
//   nvfp4_quant                           bf16 -> NVFP4 1x16 (RN)
//   mxfp8_rowwise                         MXFP8 1x32 along rows (RN or SR)
//   mx_transpose<...>                     transpose through
//                                         shared memory + MXFP8 (SR or RN)
//                                         of bf16 or dequantized NVFP4 input
//
// "End-to-End 4-Bit Training": "Low-precision formats on Blackwell" (NVFP4
// block scaling, FP32 outer scale), "Re-quantization with stochastic
// rounding" (dequantize, transpose at higher precision, SR to MXFP8), and the
// Figure 4 dataflow of the Chinese translation (row-wise and transposed SR
// quantization of the BF16 gradient).
//
// Work decomposition: every CTA owns one "window" of 128 padded rows of one
// expert group (or of one matrix of a batch) and a chunk of columns, so it
// produces whole 512-byte scale tiles, which it stages in shared memory and
// writes out with 16-byte stores.
#include "common.cuh"
#include "launch.h"

namespace nvm {

// ---------------------------------------------------------------------------
// per-tensor amax
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) amax_partial_kernel(const uint16_t *__restrict__ x,
                                                           int64_t per_batch, float *__restrict__ partial,
                                                           int nblk) {
  const int b = blockIdx.y;
  const uint4 *p = reinterpret_cast<const uint4 *>(x + (int64_t)b * per_batch);
  const int64_t n16 = per_batch >> 3;
  const int64_t st = (int64_t)nblk * 256;
  int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
  uint32_t acc0 = 0, acc1 = 0;
  for (; i + 3 * st < n16; i += 4 * st) {
    const uint4 v0 = ld_stream_v4(p + i), v1 = ld_stream_v4(p + i + st);
    const uint4 v2 = ld_stream_v4(p + i + 2 * st), v3 = ld_stream_v4(p + i + 3 * st);
    acc0 = bf16x2_absmax(acc0, bf16x2_absmax(bf16x2_absmax(v0.x, v0.y), bf16x2_absmax(v0.z, v0.w)));
    acc1 = bf16x2_absmax(acc1, bf16x2_absmax(bf16x2_absmax(v1.x, v1.y), bf16x2_absmax(v1.z, v1.w)));
    acc0 = bf16x2_absmax(acc0, bf16x2_absmax(bf16x2_absmax(v2.x, v2.y), bf16x2_absmax(v2.z, v2.w)));
    acc1 = bf16x2_absmax(acc1, bf16x2_absmax(bf16x2_absmax(v3.x, v3.y), bf16x2_absmax(v3.z, v3.w)));
  }
  for (; i < n16; i += st) {
    const uint4 v = ld_stream_v4(p + i);
    acc0 = bf16x2_absmax(acc0, bf16x2_absmax(bf16x2_absmax(v.x, v.y), bf16x2_absmax(v.z, v.w)));
  }
  float m = bf16x2_max_to_f32(bf16x2_absmax(acc0, acc1));
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, d));
  __shared__ float s_m[8];
  if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = s_m[0];
    for (int w = 1; w < 8; ++w) r = fmaxf(r, s_m[w]);
    partial[(int64_t)b * nblk + blockIdx.x] = r;
  }
}

// The amax pass over the rows x[row_src[r]], r < rows (a gathered matrix):
// one warp per row at a time, one partial maximum per block.  An index out
// of range counts as a zero row and is recorded.  cols % 8 == 0.
__global__ void __launch_bounds__(256) amax_gather_partial_kernel(const uint16_t *__restrict__ x,
                                                                  const int32_t *__restrict__ row_src,
                                                                  int64_t src_rows, int64_t rows, int64_t cols,
                                                                  float *__restrict__ partial, int nblk, int *status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t acc0 = 0, acc1 = 0;
  for (int64_t r = (int64_t)blockIdx.x * 8 + warp; r < rows; r += (int64_t)nblk * 8) {
    const int64_t sr = row_src[r];
    if (sr < 0 || sr >= src_rows) {
      if (lane == 0) record_error(status, NV_ERR_ARG);
      continue;
    }
    const uint16_t *p = x + sr * cols;
    int64_t c = (int64_t)lane * 8;
    for (; c + 256 < cols; c += 512) {
      const uint4 v0 = ld_stream_v4(p + c), v1 = ld_stream_v4(p + c + 256);
      acc0 = bf16x2_absmax(acc0, bf16x2_absmax(bf16x2_absmax(v0.x, v0.y), bf16x2_absmax(v0.z, v0.w)));
      acc1 = bf16x2_absmax(acc1, bf16x2_absmax(bf16x2_absmax(v1.x, v1.y), bf16x2_absmax(v1.z, v1.w)));
    }
    for (; c < cols; c += 256) {
      const uint4 v = ld_stream_v4(p + c);
      acc0 = bf16x2_absmax(acc0, bf16x2_absmax(bf16x2_absmax(v.x, v.y), bf16x2_absmax(v.z, v.w)));
    }
  }
  float m = bf16x2_max_to_f32(bf16x2_absmax(acc0, acc1));
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, d));
  __shared__ float s_m[8];
  if (lane == 0) s_m[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float q = s_m[0];
    for (int w = 1; w < 8; ++w) q = fmaxf(q, s_m[w]);
    partial[blockIdx.x] = q;
  }
}

// The same maximum from the tokens' own row maxima, for a token matrix no
// larger than X: a row of X is a token row, so max|X| = max over r of
// amax(x[row_src[r]]), and each token row is read once however many rows of
// X repeat it.  Stage 1: one warp per token row -> row_amax[token].
__global__ void __launch_bounds__(256) token_amax_kernel(const uint16_t *__restrict__ x, int64_t src_rows,
                                                         int64_t cols, float *__restrict__ row_amax) {
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= src_rows) return;
  const uint16_t *p = x + t * cols;
  uint32_t acc0 = 0u, acc1 = 0u;
  int64_t c = (int64_t)lane * 8;
  for (; c + 256 < cols; c += 512) {
    const uint4 v0 = ld_stream_v4(p + c), v1 = ld_stream_v4(p + c + 256);
    acc0 = bf16x2_absmax(acc0, bf16x2_absmax(bf16x2_absmax(v0.x, v0.y), bf16x2_absmax(v0.z, v0.w)));
    acc1 = bf16x2_absmax(acc1, bf16x2_absmax(bf16x2_absmax(v1.x, v1.y), bf16x2_absmax(v1.z, v1.w)));
  }
  for (; c < cols; c += 256) {
    const uint4 v = ld_stream_v4(p + c);
    acc0 = bf16x2_absmax(acc0, bf16x2_absmax(bf16x2_absmax(v.x, v.y), bf16x2_absmax(v.z, v.w)));
  }
  uint32_t m = bf16x2_absmax(acc0, acc1);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = bf16x2_absmax(m, __shfl_xor_sync(0xFFFFFFFFu, m, d));
  if (lane == 0) row_amax[t] = bf16x2_max_to_f32(m);
}

// Stage 2: one partial maximum per block of row_amax[row_src[r]]; an index
// out of range counts as a zero row and is recorded.
__global__ void __launch_bounds__(256) gather_amax_partial_kernel(const float *__restrict__ row_amax,
                                                                  const int32_t *__restrict__ row_src,
                                                                  int64_t src_rows, int64_t rows,
                                                                  float *__restrict__ partial, int nblk, int *status) {
  float m = 0.0f;
  for (int64_t r = (int64_t)blockIdx.x * 256 + threadIdx.x; r < rows; r += (int64_t)nblk * 256) {
    const int64_t sr = row_src[r];
    if (sr < 0 || sr >= src_rows) {
      record_error(status, NV_ERR_ARG);
      continue;
    }
    m = fmaxf(m, row_amax[sr]);
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, d));
  __shared__ float s_m[8];
  if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float q = s_m[0];
    for (int w = 1; w < 8; ++w) q = fmaxf(q, s_m[w]);
    partial[blockIdx.x] = q;
  }
}

// sg = amax / (6 * 448), or 1 for an all-zero tensor
__global__ void __launch_bounds__(32) outer_scale_finalize_kernel(const float *__restrict__ partial, int nblk,
                                                                  float *__restrict__ sg_out) {
  const int b = blockIdx.x;
  float m = 0.0f;
  for (int i = threadIdx.x; i < nblk; i += 32) m = fmaxf(m, partial[(int64_t)b * nblk + i]);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, d));
  if (threadIdx.x == 0) sg_out[b] = (m == 0.0f) ? 1.0f : __fdiv_rn(m, 2688.0f);
}

// Per-token outer scales ("Recipe details": one FP32 scale per token for
// activations): one warp per row, sg_r = amax_r / 2688, or 1 for an all-zero
// row.  cols % 8 == 0 (16-byte rows).
__global__ void __launch_bounds__(256) row_outer_scale_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                              int64_t cols, float *__restrict__ sg) {
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const uint16_t *p = x + r * cols;
  uint32_t m = 0u;
  for (int64_t c = (int64_t)lane * 8; c < cols; c += 256) {
    const uint4 v = ld_stream_v4(p + c);
    m = bf16x2_absmax(m, bf16x2_absmax(bf16x2_absmax(v.x, v.y), bf16x2_absmax(v.z, v.w)));
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = bf16x2_absmax(m, __shfl_xor_sync(0xFFFFFFFFu, m, d));
  if (lane == 0) {
    const float a = bf16x2_max_to_f32(m);
    sg[r] = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 2688.0f);
  }
}

// ---------------------------------------------------------------------------
// window -> rows mapping shared by the quantizers
// ---------------------------------------------------------------------------
struct Window {
  int64_t src_row0;  // first source row of the window
  int64_t rp0;       // padded row of the window's first row
  int nvalid;        // rows of the window that exist (0..128)
  int seg;           // group (grouped) or matrix (batched)
};

// grouped: windows tile the group-padded rows; batched: `wpb` windows per
// matrix of `rows` rows.  s_off/s_pad are valid when grouped.
__device__ __forceinline__ Window map_window(bool grouped, int win, int E, const int *s_off, const int *s_pad,
                                             int64_t rows, int wpb) {
  Window w;
  if (grouped) {
    const int p0 = win * 128;
    w.rp0 = p0;
    if (p0 >= s_pad[E]) {
      w.src_row0 = 0; w.nvalid = 0; w.seg = E;
    } else {
      const int e = find_group(s_pad, E, p0);
      w.seg = e;
      w.src_row0 = (int64_t)s_off[e] + (p0 - s_pad[e]);
      const int64_t left = (int64_t)s_off[e + 1] - w.src_row0;
      w.nvalid = left < 128 ? (int)left : 128;
    }
  } else {
    const int b = win / wpb, wb = win - b * wpb;
    w.seg = b;
    w.src_row0 = (int64_t)b * rows + (int64_t)wb * 128;
    w.rp0 = ((int64_t)b * wpb + wb) * 128;
    const int64_t left = rows - (int64_t)wb * 128;
    w.nvalid = left < 128 ? (int)left : 128;
  }
  return w;
}

// Shared-memory group tables.  E == 0 with `single` means one group of all
// rows (offsets {0, rows}) built without reading global memory.
struct GroupSmem {
  int flag;
  int off[kMaxGroups + 1];
  int pad[kMaxGroups + 1];
};

__device__ __forceinline__ bool setup_groups(GroupSmem &g, const int32_t *go, int &E, int64_t rows, int *status) {
  if (go == nullptr) {  // one group of all rows
    if (threadIdx.x == 0) {
      g.off[0] = 0; g.off[1] = (int)rows;
      g.pad[0] = 0; g.pad[1] = (int)((rows + 127) & ~127LL);
    }
    E = 1;
    __syncthreads();
    return true;
  }
  return load_groups(go, E, rows, g.off, g.pad, &g.flag, status);
}

// The CTA's window in the grouped layout, worked out by warp 0 alone: it
// reads the group offsets, checks them as load_groups does (offsets[0] == 0,
// offsets[E] == rows, non-decreasing, within [0, rows]; otherwise
// NV_ERR_OFFSETS is recorded and every thread gets false), scans the
// 128-padded group sizes and finds the group holding padded row 128 * win
// (the result of map_window); the other warps read it after one barrier
// instead of repeating the setup and a binary search each.  go == nullptr:
// one group of all rows.  Every thread of the CTA must call it.
__device__ __forceinline__ bool grouped_window(const int32_t *__restrict__ go, int E, int64_t rows, int win,
                                               int *status, Window &w) {
  __shared__ Window s_win;
  __shared__ int s_bad;
  if (threadIdx.x < 32) {
    const int lane = (int)threadIdx.x;
    const int p0 = win * 128;
    if (go == nullptr) E = 1;
    bool bad = false, found = false;
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int lo = 0, hi = 0;
      if (e < E) {
        lo = go ? go[e] : 0;
        hi = go ? go[e + 1] : (int)rows;
        bad |= lo < 0 || hi < lo || (int64_t)hi > rows || (e == 0 && lo != 0) || (e == E - 1 && (int64_t)hi != rows);
      }
      const int sz = (hi - lo + 127) & ~127;  // 0 past the last group
      int incl = sz;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += n;
      }
      const int start = carry + incl - sz;
      const bool hit = sz > 0 && p0 >= start && p0 < start + sz;
      if (hit) {
        Window t;
        t.rp0 = p0;
        t.seg = e;
        t.src_row0 = (int64_t)lo + (p0 - start);
        const int64_t left = (int64_t)hi - t.src_row0;
        t.nvalid = left < 128 ? (int)left : 128;
        s_win = t;
      }
      found |= __any_sync(0xFFFFFFFFu, hit);
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    bad = __any_sync(0xFFFFFFFFu, bad);
    if (lane == 0) {
      s_bad = bad ? 1 : 0;
      if (bad) record_error(status, NV_ERR_OFFSETS);
      if (!found) {  // a window past the last group's padded rows
        Window t;
        t.rp0 = p0;
        t.seg = E;
        t.src_row0 = 0;
        t.nvalid = 0;
        s_win = t;
      }
    }
  }
  __syncthreads();
  if (s_bad) return false;
  w = s_win;
  return true;
}

// ---------------------------------------------------------------------------
// NVFP4 quantization, one CTA = 128 padded rows x 256 columns
// ---------------------------------------------------------------------------
struct NvQuantArgs {
  const uint16_t *x;
  int64_t rows, cols;
  const int32_t *groups;  // non-null: grouped scale layout (batch == 1)
  int E;
  int wpb;                // windows per matrix (batched)
  const float *sg;        // [batch]
  const float *sg_rows;   // non-null: one outer scale per row (per token) instead
  int four_six;           // Four Over Six block rule (nvfp4_block46)
  uint8_t *codes, *scales;
  int64_t ka;             // scale tiles per padded row tile = ceil(cols / 64)
  int *status;
};

// inv_tab: when the outer scale is the same for every block of the CTA, the
// 127 values fp32(1 / fp32(s * sg)) of the E4M3 codes (0 for code 0), read
// instead of computing the reciprocal per block (the same bits)
__device__ __forceinline__ void nvfp4_block(const uint4 &a, const uint4 &b, float sg, float den6, uint2 &codes,
                                            uint32_t &scode, const float *inv_tab = nullptr) {
  uint32_t m = bf16x2_absmax(bf16x2_absmax(a.x, a.y), bf16x2_absmax(a.z, a.w));
  m = bf16x2_absmax(m, bf16x2_absmax(bf16x2_absmax(b.x, b.y), bf16x2_absmax(b.z, b.w)));
  const float bamax = bf16x2_max_to_f32(m);
  scode = cvt_e4m3_rn(__fdiv_rn(bamax, den6));
  float inv;
  if (inv_tab) {
    inv = inv_tab[scode];
  } else {
    const float s = e4m3_to_f32(scode);
    inv = (s == 0.0f) ? 0.0f : __frcp_rn(__fmul_rn(s, sg));
  }
  codes.x = cvt_e2m1x8(__fmul_rn(bf16_lo(a.x), inv), __fmul_rn(bf16_hi(a.x), inv), __fmul_rn(bf16_lo(a.y), inv),
                       __fmul_rn(bf16_hi(a.y), inv), __fmul_rn(bf16_lo(a.z), inv), __fmul_rn(bf16_hi(a.z), inv),
                       __fmul_rn(bf16_lo(a.w), inv), __fmul_rn(bf16_hi(a.w), inv));
  codes.y = cvt_e2m1x8(__fmul_rn(bf16_lo(b.x), inv), __fmul_rn(bf16_hi(b.x), inv), __fmul_rn(bf16_lo(b.y), inv),
                       __fmul_rn(bf16_hi(b.y), inv), __fmul_rn(bf16_lo(b.z), inv), __fmul_rn(bf16_hi(b.z), inv),
                       __fmul_rn(bf16_lo(b.w), inv), __fmul_rn(bf16_hi(b.w), inv));
}

__device__ __forceinline__ void nvfp4_block46(const uint4 &a, const uint4 &b, float sg, uint2 &codes,
                                              uint32_t &scode);

// nvfp4_block with the division bamax / den6 read from a table and the
// element multiplies packed two at a time; the same bits.  qtab[m] holds
// fp32((1 + m / 128) / den6): for a normal bf16 block maximum
// (1 + m / 128) 2^e, fp32(bamax / den6) = qtab[m] 2^e exactly while the
// quotient is a normal fp32 number (scaling by a power of two commutes with
// rounding there), and below that range or at overflow both forms give the
// same E4M3 code (0, or the 448 saturation).  qtab[128 + m] holds the
// quotient itself for the subnormal (and zero) bf16 maximum m 2^-133, read
// with multiplier 1.  inv_tab as in nvfp4_block.
__device__ __forceinline__ void mul2_rn(float a, float b, float m, float &ra, float &rb);
__device__ __forceinline__ void nvfp4_block_tab(const uint4 &a, const uint4 &b, const float *qtab,
                                                const float *inv_tab, uint2 &codes, uint32_t &scode) {
  uint32_t m = bf16x2_absmax(bf16x2_absmax(a.x, a.y), bf16x2_absmax(a.z, a.w));
  m = bf16x2_absmax(m, bf16x2_absmax(bf16x2_absmax(b.x, b.y), bf16x2_absmax(b.z, b.w)));
  const uint32_t u = max(m & 0x7FFFu, (m >> 16) & 0x7FFFu);  // |block max| as bf16 bits (signs meaningless)
  const uint32_t e = u & 0x7F80u;
  const bool sub = e == 0u;
  const float q = __fmul_rn(qtab[(u & 0x7Fu) | (sub ? 128u : 0u)], __uint_as_float(sub ? 0x3F800000u : e << 16));
  scode = cvt_e4m3_rn(q);
  const float inv = inv_tab[scode];
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float f[16];
#pragma unroll
  for (int k = 0; k < 8; ++k) mul2_rn(bf16_lo(w[k]), bf16_hi(w[k]), inv, f[2 * k], f[2 * k + 1]);
  codes.x = cvt_e2m1x8(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]);
  codes.y = cvt_e2m1x8(f[8], f[9], f[10], f[11], f[12], f[13], f[14], f[15]);
}

// the reciprocal table of nvfp4_block for one outer scale (threads 0..127)
__device__ __forceinline__ void fill_inv_table(float *tab, float sg) {
  if (threadIdx.x < 128) {
    const float s = e4m3_to_f32(threadIdx.x);
    tab[threadIdx.x] = (s == 0.0f) ? 0.0f : __frcp_rn(__fmul_rn(s, sg));  // the formula of nvfp4_block
  }
}

__global__ void __launch_bounds__(256) nvfp4_quant_kernel(NvQuantArgs A) {
  __shared__ __align__(16) uint8_t s_sc[4 * 512];
  const bool grouped = A.groups != nullptr;
  Window w;
  if (grouped) {
    if (!grouped_window(A.groups, A.E, A.rows, blockIdx.y, A.status, w)) return;
  } else {
    w = map_window(false, blockIdx.y, 0, nullptr, nullptr, A.rows, A.wpb);
  }
  const float sg = A.sg_rows ? 1.0f : A.sg[grouped ? 0 : w.seg];
  const float den6 = __fmul_rn(6.0f, sg);
  __shared__ float s_inv[128];
  fill_inv_table(s_inv, sg);

  reinterpret_cast<uint2 *>(s_sc)[threadIdx.x] = make_uint2(0u, 0u);
  __syncthreads();

  const int KB = (int)(A.cols >> 4);
  const int kb0 = blockIdx.x * 16;
  const int nkb = min(16, KB - kb0);
  // four blocks of 16 per thread per phase, two phases
#pragma unroll
  for (int ph = 0; ph < 2; ++ph) {
    uint4 va[4], vb[4];
    bool ok[4];
    int64_t off[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = (ph * 4 + u) * 256 + threadIdx.x;
      const int i = q >> 4, kbl = q & 15;
      ok[u] = (i < w.nvalid) && (kbl < nkb);
      off[u] = (w.src_row0 + i) * A.cols + (int64_t)(kb0 + kbl) * 16;
      if (ok[u]) {
        va[u] = ld_stream_v4(A.x + off[u]);
        vb[u] = ld_stream_v4(A.x + off[u] + 8);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (!ok[u]) continue;
      const int q = (ph * 4 + u) * 256 + threadIdx.x;
      const int i = q >> 4, kbl = q & 15;
      uint2 c;
      uint32_t sc;
      if (A.sg_rows) {
        const float sgi = A.sg_rows[w.src_row0 + i];
        nvfp4_block(va[u], vb[u], sgi, __fmul_rn(6.0f, sgi), c, sc);
      } else if (A.four_six) {
        nvfp4_block46(va[u], vb[u], sg, c, sc);
      } else {
        nvfp4_block(va[u], vb[u], sg, den6, c, sc, s_inv);
      }
      *reinterpret_cast<uint2 *>(A.codes + (off[u] >> 1)) = c;
      s_sc[(kbl >> 2) * 512 + atom_pos(i, kbl)] = (uint8_t)sc;
    }
  }
  __syncthreads();
  // write the (up to) four 512-byte scale tiles of this window / chunk
  if (threadIdx.x < 128) {
    const int a = threadIdx.x >> 5, part = threadIdx.x & 31;
    const int64_t tile_col = kb0 / 4 + a;
    if (tile_col < A.ka) {
      const int64_t dst = ((w.rp0 >> 7) * A.ka + tile_col) * 512 + part * 16;
      *reinterpret_cast<uint4 *>(A.scales + dst) = reinterpret_cast<const uint4 *>(s_sc + a * 512)[part];
    }
  }
}

// ---------------------------------------------------------------------------
// MXFP8 along rows: one CTA = 128 padded rows x 256 columns (8 blocks of 32)
// ---------------------------------------------------------------------------
struct MxRowArgs {
  const uint16_t *x;
  int64_t rows, cols;
  const int32_t *groups;
  int E;
  int sr;
  uint64_t seed, offset;
  PhiloxRoundKeys rk;  // round keys of `seed`
  uint8_t *codes, *scales;
  int64_t ka;  // ceil(cols / 128)
  int *status;
};

// RN of 8 consecutive elements with multiplier `mult`
__device__ __forceinline__ uint2 mx_rn8(const float (&v)[8], float mult) {
  const uint32_t p0 = cvt_e4m3x2_rn(__fmul_rn(v[0], mult), __fmul_rn(v[1], mult));
  const uint32_t p1 = cvt_e4m3x2_rn(__fmul_rn(v[2], mult), __fmul_rn(v[3], mult));
  const uint32_t p2 = cvt_e4m3x2_rn(__fmul_rn(v[4], mult), __fmul_rn(v[5], mult));
  const uint32_t p3 = cvt_e4m3x2_rn(__fmul_rn(v[6], mult), __fmul_rn(v[7], mult));
  return make_uint2(p0 | (p1 << 16), p2 | (p3 << 16));
}

// SR of 8 consecutive bf16 elements of a row (one uint4) with the power-of-two
// multiplier whose bf16 bits are `m`; w0 and w1 are the Philox words of their
// four pairs (pairs 0,1 in w0, pairs 2,3 in w1)
__device__ __forceinline__ uint2 mx_sr8(const uint4 &q, uint16_t m, uint32_t w0, uint32_t w1) {
  return make_uint2(cvt_e4m3x4_sr(bf16_lo_times(q.x, m), bf16_hi_times(q.x, m), bf16_lo_times(q.y, m),
                                  bf16_hi_times(q.y, m), ~w0),
                    cvt_e4m3x4_sr(bf16_lo_times(q.z, m), bf16_hi_times(q.z, m), bf16_lo_times(q.w, m),
                                  bf16_hi_times(q.w, m), ~w1));
}

__device__ __forceinline__ void unpack8(const uint4 &q, float (&v)[8]) {
  v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
  v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
}

__global__ void __launch_bounds__(256) mxfp8_rowwise_kernel(const __grid_constant__ MxRowArgs A) {
  __shared__ __align__(16) uint8_t s_sc[2 * 512];
  Window w;
  if (!grouped_window(A.groups, A.E, A.rows, blockIdx.y, A.status, w)) return;
  reinterpret_cast<uint32_t *>(s_sc)[threadIdx.x] = 0u;
  __syncthreads();
  const int KB = (int)(A.cols >> 5);
  const int kb0 = blockIdx.x * 8;
  const int nkb = min(8, KB - kb0);
#pragma unroll 1
  for (int it = 0; it < 4; ++it) {
    const int q = it * 256 + threadIdx.x;
    const int i = q >> 3, kbl = q & 7;
    if (i >= w.nvalid || kbl >= nkb) continue;
    const int64_t e0 = (w.src_row0 + i) * A.cols + (int64_t)(kb0 + kbl) * 32;
    uint4 raw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) raw[k] = ld_stream_v4(A.x + e0 + 8 * k);
    uint32_t m = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) m = bf16x2_absmax(m, bf16x2_absmax(bf16x2_absmax(raw[k].x, raw[k].y), bf16x2_absmax(raw[k].z, raw[k].w)));
    float mult;
    const uint32_t sc = e8m0_scale(bf16x2_max_to_f32(m), &mult);
    uint2 out[4];
    // pair keys (e0 / 2) .. (e0 / 2) + 15: two Philox calls, one word per 4 elements
    uint4 bits0 = make_uint4(0, 0, 0, 0), bits1 = make_uint4(0, 0, 0, 0);
    if (A.sr) {
      bits0 = philox_bits8_rk((uint64_t)(e0 >> 4), A.offset, A.rk);
      bits1 = philox_bits8_rk((uint64_t)(e0 >> 4) + 1, A.offset, A.rk);
    }
    const uint16_t mb = pow2_bf16_bits(mult);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (A.sr) {
        const uint4 &b = k < 2 ? bits0 : bits1;
        out[k] = (k & 1) ? mx_sr8(raw[k], mb, b.z, b.w) : mx_sr8(raw[k], mb, b.x, b.y);
      } else {
        float v[8];
        unpack8(raw[k], v);
        out[k] = mx_rn8(v, mult);
      }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(A.codes + e0);
    dst[0] = make_uint4(out[0].x, out[0].y, out[1].x, out[1].y);
    dst[1] = make_uint4(out[2].x, out[2].y, out[3].x, out[3].y);
    s_sc[(kbl >> 2) * 512 + atom_pos(i, kbl)] = (uint8_t)sc;
  }
  __syncthreads();
  if (threadIdx.x < 64) {
    const int a = threadIdx.x >> 5, part = threadIdx.x & 31;
    const int64_t tile_col = kb0 / 4 + a;
    if (tile_col < A.ka) {
      const int64_t dst = ((w.rp0 >> 7) * A.ka + tile_col) * 512 + part * 16;
      *reinterpret_cast<uint4 *>(A.scales + dst) = reinterpret_cast<const uint4 *>(s_sc + a * 512)[part];
    }
  }
}

// ---------------------------------------------------------------------------
// Transposed MXFP8 (the SR re-quantization of saved NVFP4 operands, and the
// WGRAD operand of the gradient quantizer): one CTA = 128 padded
// source rows (one window) x 128 source columns.  Three sources (kMode):
//   kSrcBf16        bf16 -> MXFP8 SR/RN, transposed (+ optional row-wise)
//   kSrcNvfp4       NVFP4 codes + scales + outer scale -> dequantize ->
//                   transposed SR to MXFP8 (the re-quantization)
//   kSrcBf16ToNvfp4 bf16 -> NVFP4 (codes, scales; the quantizer's block rule)
//                   and, from the codes just made, the same re-quantization:
//                   both outputs of nvfp4_quantize + dequant_transpose_
//                   requant_sr in one pass over the source
// kGather (NVFP4 output, per-tensor scale): row r of the window is source
// row row_src[r] -- bf16 token rows (kSrcBf16ToNvfp4), or the NVFP4 codes
// and per-row block scales of already quantized tokens (kSrcNvfp4, which
// then also copies them to the routed rows' NVFP4 layout).  A window without
// data (grouped padding past the last group) only writes zero scale tiles.
//   phase 1  stream the tile into shared memory as 16-bit values: bf16 input
//            as is, NVFP4 input as the exact f16 products e2m1 * e4m3 (at most
//            6 significant bits, inside the f16 range); optionally emit the
//            row-wise MXFP8 output (bf16 input)
//   phase 2  per output row (= source column) and 32-token block: amax on
//            packed halves, E8M0 scale, SR (bits drawn at the source index) or
//            RN -> bytes
//            -> 128-byte output rows, stored from registers (a warp writes
//            one whole row per store instruction)
//   phase 3  write the 512-byte scale tiles
// The value tile keeps 16-byte chunk c8 of row i at chunk c8 ^ ((i >> 2) & 7),
// which makes both the row-wise fill and the 4-tokens-per-lane column reads
// bank-conflict free.
// ---------------------------------------------------------------------------
enum { kSrcBf16 = 0, kSrcNvfp4 = 1, kSrcBf16ToNvfp4 = 2 };

struct MxTArgs {
  // input
  const uint16_t *x;                 // bf16 source (kSrcBf16, kSrcBf16ToNvfp4)
  const int32_t *row_src;            // kSrcBf16ToNvfp4: row r of the source is x row row_src[r] (null: r)
  int64_t src_rows;                  // rows of x when row_src is given
  const uint8_t *nv_codes;           // NVFP4 source (kSrcNvfp4)
  const uint8_t *nv_scales;
  const float *nv_sg;                // outer scale: [batch] (batched) or [1]
  const float *nv_sg_rows;           // per-token outer scales [rows] (kRows kernels)
  // NVFP4 output (kSrcBf16ToNvfp4)
  uint8_t *nv_codes_out, *nv_scales_out;
  int64_t nv_ka;                     // NVFP4 scale tiles per 128 rows = cols / 64
  int64_t rows, cols;                // rows per matrix (batched) or total rows
  const int32_t *groups;             // grouped mode when non-null or `single`
  int E;
  int grouped;                       // 1: grouped/single-group layouts, 0: batched
  int wpb;                           // windows per matrix (batched)
  int sr;
  uint64_t seed, off_t, off_row;
  PhiloxRoundKeys rk;                // round keys of `seed`
  // transposed output
  uint8_t *out_codes, *out_scales;
  int64_t out_stride;                // P_cap (grouped)
  int64_t out_ka;                    // scale tiles per 128 output rows
  // row-wise output (bf16 source only; may be null)
  uint8_t *row_codes, *row_scales;
  int64_t row_ka;
  int *status;
};

constexpr int kTileSmem = 128 * 256;                 // 128 rows x 128 16-bit values, swizzled
constexpr int kNvStage = 128 * 64 + 1024;            // NVFP4 source: staged codes and two scale tiles

__device__ __forceinline__ int chunk_of(int i, int c8) { return c8 ^ ((i >> 2) & 7); }
// The swizzle of the NVFP4-source kernel's 8-tokens-per-lane column pass:
// chunk c of row i at (c even: c / 2, odd: 8 + c / 2) XOR ((i >> 3) & 7).
// The product fill (eight lanes, one row's even or odd chunks) and the
// column reads (eight lanes, one chunk of rows 8 apart) both land on eight
// distinct bank groups.
__device__ __forceinline__ int chunk_of8(int i, int c) { return ((c & 1) << 3) | ((c >> 1) ^ ((i >> 3) & 7)); }
template <bool kT8>
__device__ __forceinline__ int tile_chunk(int i, int c) { return kT8 ? chunk_of8(i, c) : chunk_of(i, c); }
__device__ __forceinline__ uint32_t word_of(const uint4 &v, int p) {
  return p == 0 ? v.x : p == 1 ? v.y : p == 2 ? v.z : v.w;
}

// eight E2M1 codes (one 32-bit word, element k in nibble k) -> four f16x2
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// max(|a|, |b|) per f16 half; the sign bits of the result are meaningless
__device__ __forceinline__ uint32_t habsmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// (fp32(a * m), fp32(b * m)) with one packed fp32x2 multiply (each lane
// rounded to nearest even, exactly as two separate multiplies)
__device__ __forceinline__ void mul2_rn(float a, float b, float m, float &ra, float &rb) {
  uint64_t x, mm, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
  asm("mov.b64 %0, {%1, %1};" : "=l"(mm) : "f"(m));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(x), "l"(mm));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(ra), "=f"(rb) : "l"(d));
}
__device__ __forceinline__ float f16_lo(uint32_t w) {
  float f;
  asm("{ .reg .f16 lo, hi;\n\t mov.b32 {lo, hi}, %1;\n\t cvt.f32.f16 %0, lo; }" : "=f"(f) : "r"(w));
  return f;
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
  float f;
  asm("{ .reg .f16 lo, hi;\n\t mov.b32 {lo, hi}, %1;\n\t cvt.f32.f16 %0, hi; }" : "=f"(f) : "r"(w));
  return f;
}
// E4M3 code -> f16x2 (s, s), exact
__device__ __forceinline__ uint32_t e4m3_to_f16x2_dup(uint32_t code) {
  uint32_t h2;
  const uint16_t c16 = (uint16_t)((code & 0xFFu) * 0x0101u);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c16));
  return h2;
}

// Squared quantization error of one block in fp32, in element order:
// d_i = fp32(fp32(e2m1_i * s) * sg), e_i = fp32(x_i - d_i), acc = fp32(acc + fp32(e_i^2))
// (every operation rounded on its own: no fused multiply-add).
__device__ __forceinline__ float nvfp4_block_sq_err(const uint4 &a, const uint4 &b, uint2 codes, float s, float sg) {
  uint32_t h[8];
  e2m1x8_to_f16x2(codes.x, reinterpret_cast<uint32_t(&)[4]>(h[0]));
  e2m1x8_to_f16x2(codes.y, reinterpret_cast<uint32_t(&)[4]>(h[4]));
  const uint32_t xw[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float acc = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float d0 = __fmul_rn(__fmul_rn(f16_lo(h[k]), s), sg);
    const float d1 = __fmul_rn(__fmul_rn(f16_hi(h[k]), s), sg);
    const float e0 = __fsub_rn(bf16_lo(xw[k]), d0);
    const float e1 = __fsub_rn(bf16_hi(xw[k]), d1);
    acc = __fadd_rn(acc, __fmul_rn(e0, e0));
    acc = __fadd_rn(acc, __fmul_rn(e1, e1));
  }
  return acc;
}

// Four Over Six: the block quantized with its maximum mapped to 6 (the plain
// rule) and to 4, under the same outer scale; the smaller squared error wins,
// ties keep 6
__device__ __forceinline__ void nvfp4_block46(const uint4 &a, const uint4 &b, float sg, uint2 &codes,
                                              uint32_t &scode) {
  uint2 c6, c4;
  uint32_t s6, s4;
  nvfp4_block(a, b, sg, __fmul_rn(6.0f, sg), c6, s6);
  nvfp4_block(a, b, sg, __fmul_rn(4.0f, sg), c4, s4);
  const float e6 = nvfp4_block_sq_err(a, b, c6, e4m3_to_f32(s6), sg);
  const float e4 = nvfp4_block_sq_err(a, b, c4, e4m3_to_f32(s4), sg);
  const bool take4 = e4 < e6;
  codes = take4 ? c4 : c6;
  scode = take4 ? s4 : s6;
}

// the 16 exact f16 products e2m1 * e4m3 of one (row i, 16-column block kb)
// unit into the swizzled 16-bit tile
template <bool kT8 = false>
__device__ __forceinline__ void store_f16_products(uint8_t *s_in, int i, int kb, uint2 codes, uint32_t scale) {
  const uint32_t s2 = e4m3_to_f16x2_dup(scale);
  uint32_t h0[4], h1[4];
  e2m1x8_to_f16x2(codes.x, h0);
  e2m1x8_to_f16x2(codes.y, h1);
  uint4 *row = reinterpret_cast<uint4 *>(s_in + i * 256);
  row[tile_chunk<kT8>(i, 2 * kb)] =
      make_uint4(hmul2_u32(h0[0], s2), hmul2_u32(h0[1], s2), hmul2_u32(h0[2], s2), hmul2_u32(h0[3], s2));
  row[tile_chunk<kT8>(i, 2 * kb + 1)] =
      make_uint4(hmul2_u32(h1[0], s2), hmul2_u32(h1[1], s2), hmul2_u32(h1[2], s2), hmul2_u32(h1[3], s2));
}

// 16-byte asynchronous global -> shared copy (L2 only); `bytes` (0 or 16) are
// read and the rest is zero-filled
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(bytes)
               : "memory");
}
// the same for 4 bytes (`bytes` 0 or 4)
__device__ __forceinline__ void cp_async4(void *dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(bytes)
               : "memory");
}

// The window's bf16 tile [128 rows][128 columns] straight into the swizzled
// 16-bit layout with cp.async: 128 bytes per thread in flight without
// registers; rows past the window's data are zero-filled.  Waits for the
// thread's own copies; the caller's barrier makes the tile visible.
// kGather: row r of the window is source row row_src[r].  kWarpRows: warp w
// stages rows 32 u + 4 w + j (u, j < 4), the rows of its units in the
// row-wise NVFP4 pass, so that a __syncwarp makes them visible to it.
template <bool kGather, bool kWarpRows = false>
__device__ __forceinline__ void stage_bf16_tile(const MxTArgs &A, const Window &w, int64_t col0, uint8_t *s_in) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int q = k * 256 + (int)threadIdx.x;
    int i = q >> 4, c16 = q & 15;
    if (kWarpRows) {  // 16 rows x 16 chunks per warp, two whole rows per warp instruction
      const int m = k * 32 + (int)(threadIdx.x & 31), rho = m >> 4;
      i = 32 * (rho >> 2) + 4 * (int)(threadIdx.x >> 5) + (rho & 3);
      c16 = m & 15;
    }
    bool ok = i < w.nvalid;
    int64_t row = w.src_row0 + i;
    if (kGather && ok) {  // a row index out of range reads as zeros and is recorded
      row = A.row_src[row];
      if (row < 0 || row >= A.src_rows) {
        record_error(A.status, NV_ERR_ARG);
        ok = false;
      }
    }
    const uint16_t *src = ok ? A.x + row * A.cols + col0 + c16 * 8 : A.x;
    cp_async16(s_in + i * 256 + chunk_of(i, c16) * 16, src, ok ? 16u : 0u);
  }
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
}

// CTAs per SM: five (48 registers) for the bf16 -> NVFP4 kernels, where the
// extra warps hide more of the barrier and load waits (about 3% faster than
// four); four (64 registers) for the bf16 gradient kernel, for which five
// measured no faster, and for the NVFP4-source kernel, whose
// 8-tokens-per-lane column pass needs them; three for the per-token
// kernels, which spill at more
template <int kMode, bool kRows>
constexpr int mx_t_min_blocks() { return kRows ? 3 : (kMode == 0 || kMode == 1) ? 4 : 5; }

template <int kMode, bool kRows = false, bool k46 = false, bool kGather = false>
__global__ void __launch_bounds__(256, mx_t_min_blocks<kMode, kRows>()) mx_transpose_kernel(
    const __grid_constant__ MxTArgs A) {
  constexpr bool kNvfp4 = kMode != kSrcBf16;  // phase 2 on exact f16 products of NVFP4 values
  static_assert(!kRows || kNvfp4, "per-token outer scales apply to NVFP4 sources");
  static_assert(!kGather || (kMode != kSrcBf16 && !kRows && !k46), "gathered rows: NVFP4 output, per-tensor scale");
  // the routed rows' NVFP4 codes and scales are written too (from the bf16
  // source, or copied from the gathered token codes)
  constexpr bool kNvOut = kMode == kSrcBf16ToNvfp4 || kGather;
  // the NVFP4-source kernel (per-tensor scale) runs the column pass with 8
  // tokens per lane, on its own tile swizzle (chunk_of8)
  constexpr bool kT8 = kMode == kSrcNvfp4 && !kRows;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ __align__(16) uint8_t s_tsc[512];   // transposed scale tile
  __shared__ __align__(16) uint8_t s_rsc[512];   // row-wise scale tile
  __shared__ __align__(16) uint8_t s_nvsc[kNvOut ? 1024 : 16];  // NVFP4 scale tiles
  uint8_t *s_stage = smem;                                           // NVFP4 source staging (kSrcNvfp4)
  uint8_t *s_in = smem + (kMode == kSrcNvfp4 ? kNvStage : 0);         // [128][256 B] 16-bit values

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the row-wise scale tile (bf16 source, always grouped) keeps zeros for rows
  // without data; the barrier of the group lookup orders this clearing before
  // any phase-1 write
  if (kMode == kSrcBf16 && tid < 128) reinterpret_cast<uint32_t *>(s_rsc)[tid] = 0u;
  Window w;
  if (A.grouped) {
    if (!grouped_window(A.groups, A.E, A.rows, blockIdx.y, A.status, w)) return;
  } else {
    w = map_window(false, blockIdx.y, 0, nullptr, nullptr, A.rows, A.wpb);
  }
  const int64_t col0 = (int64_t)blockIdx.x * 128;

  // output addressing: transposed codes [source column][token], scale tile
  int64_t out_base, out_stride, tile_idx;
  if (A.grouped) {
    out_base = col0 * A.out_stride + w.rp0;
    out_stride = A.out_stride;
    tile_idx = (col0 >> 7) * A.out_ka + (w.rp0 >> 7);
  } else {
    const int b = w.seg;
    const int64_t wb = w.rp0 / 128 - (int64_t)b * A.wpb;
    out_base = ((int64_t)b * A.cols + col0) * A.rows + wb * 128;
    out_stride = A.rows;
    const int64_t cpad = (A.cols + 127) & ~127LL;
    tile_idx = (((int64_t)b * cpad + col0) >> 7) * A.out_ka + wb;
  }
  if (w.nvalid == 0) {
    // a window without data (grouped padding past the last group): zero
    // scale tiles, no codes (w is the same for every thread: no barrier is
    // left unmatched)
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    if (tid < 32) {
      reinterpret_cast<uint4 *>(A.out_scales + tile_idx * 512)[tid] = z;
    } else if (tid < 64 && A.row_codes != nullptr) {
      reinterpret_cast<uint4 *>(A.row_scales + ((w.rp0 >> 7) * A.row_ka + (col0 >> 7)) * 512)[tid - 32] = z;
    } else if (kNvOut && tid >= 64 && tid < 128) {
      reinterpret_cast<uint4 *>(A.nv_scales_out + ((w.rp0 >> 7) * A.nv_ka + (col0 >> 6)) * 512)[tid - 64] = z;
    }
    return;
  }
  const float sg = kNvfp4 && !kRows ? A.nv_sg[A.grouped ? 0 : w.seg] : 1.0f;

  // ---- phase 1 --------------------------------------------------------------
  if (!kNvfp4) {
    // the warp's own rows (a __syncwarp): the row-wise pass reads only them;
    // the barrier after it makes the whole tile visible to the column pass
    stage_bf16_tile<false, true>(A, w, col0, s_in);
    __syncwarp();
    // row-wise output: items of 16 columns (32 bytes) of one row; a row-wise
    // MXFP8 block of 32 is two neighbouring lanes, and one Philox call covers
    // an item's 8 pairs
    if (A.row_codes != nullptr) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = u * 256 + tid;
        const int i = q >> 3, c16 = q & 7;
        const uint4 *row = reinterpret_cast<const uint4 *>(s_in + i * 256);
        const uint4 r0 = row[chunk_of(i, 2 * c16)], r1 = row[chunk_of(i, 2 * c16 + 1)];
        const bool valid = i < w.nvalid;
        const int64_t e0 = (w.src_row0 + i) * A.cols + col0 + c16 * 16;
        uint32_t m = bf16x2_absmax(bf16x2_absmax(r0.x, r0.y), bf16x2_absmax(r0.z, r0.w));
        m = bf16x2_absmax(m, bf16x2_absmax(bf16x2_absmax(r1.x, r1.y), bf16x2_absmax(r1.z, r1.w)));
        m = bf16x2_absmax(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        if (valid) {
          float mult;
          const uint32_t sc = e8m0_scale(bf16x2_max_to_f32(m), &mult);
          uint2 o0, o1;
          if (A.sr) {
            const uint4 b = philox_bits8_rk((uint64_t)(e0 >> 4), A.off_row, A.rk);  // pair keys e0/2 .. e0/2+7
            const uint16_t mb = pow2_bf16_bits(mult);
            o0 = mx_sr8(r0, mb, b.x, b.y);
            o1 = mx_sr8(r1, mb, b.z, b.w);
          } else {
            float v0[8], v1[8];
            unpack8(r0, v0);
            unpack8(r1, v1);
            o0 = mx_rn8(v0, mult);
            o1 = mx_rn8(v1, mult);
          }
          *reinterpret_cast<uint4 *>(A.row_codes + e0) = make_uint4(o0.x, o0.y, o1.x, o1.y);
          if ((c16 & 1) == 0) s_rsc[atom_pos(i, c16 >> 1)] = (uint8_t)sc;
        }
      }
    }
  } else if (kMode == kSrcNvfp4) {
    // NVFP4: the window's codes [128 rows][64 bytes] and its two 512-byte
    // scale tiles go through cp.async into the staging area, then each (row,
    // 16-column block) unit is decoded to exact f16 products e2m1 * e4m3.
    // kGather: row i is token row_src[src_row0 + i] of a token matrix in the
    // batched layout; thread (i = tid / 2, half h = tid % 2) stages that
    // row's 32 code bytes of half h and its four block scales of half h (one
    // 4-byte word of the token's scale tile h), rows per unit instead of the
    // two tiles, and a CTA barrier follows (the fill's rows are other warps');
    // otherwise each warp stages exactly what its own fill reads
    uint8_t *st_codes = s_stage, *st_sc = s_stage + 128 * 64;
    const int64_t half_cols = A.cols >> 1;
    if (kGather) {
      const int i = tid >> 1, h = tid & 1;
      bool ok = i < w.nvalid;
      int64_t t = 0;
      if (ok) {  // a row index out of range reads as zeros and is recorded
        t = A.row_src[w.src_row0 + i];
        if (t < 0 || t >= A.src_rows) {
          record_error(A.status, NV_ERR_ARG);
          ok = false;
        }
      }
      const uint8_t *src = ok ? A.nv_codes + t * half_cols + (col0 >> 1) + h * 32 : A.nv_codes;
      cp_async16(st_codes + i * 64 + h * 32, src, ok ? 16u : 0u);
      cp_async16(st_codes + i * 64 + h * 32 + 16, ok ? src + 16 : A.nv_codes, ok ? 16u : 0u);
      const int64_t ka_src = A.cols >> 6;
      const uint8_t *ssrc =
          ok ? A.nv_scales + ((t >> 7) * ka_src + (col0 >> 6) + h) * 512 + atom_pos((int)(t & 127), 0) : A.nv_scales;
      cp_async4(st_sc + i * 8 + h * 4, ssrc, ok ? 4u : 0u);
    } else {
      // warp w: the codes of rows 32 u + 4 w + j (u, j < 4), the rows of its
      // units in the product fill below, and their scales: bytes 64 w ..
      // 64 w + 63 of both scale tiles (row i's four scales sit at (i % 32) 16
      // + (i / 32) 4), so that a __syncwarp makes them visible to it
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int unit = k * 32 + lane, rho = unit >> 2;
        const int i = 32 * (rho >> 2) + 4 * warp + (rho & 3), part = unit & 3;
        const bool ok = i < w.nvalid;
        const uint8_t *src = ok ? A.nv_codes + (w.src_row0 + i) * half_cols + (col0 >> 1) + part * 16 : A.nv_codes;
        cp_async16(st_codes + i * 64 + part * 16, src, ok ? 16u : 0u);
      }
      if (lane < 8) {
        const int64_t ka_src = (A.cols + 63) >> 6;
        const int64_t tile0 = (w.rp0 >> 7) * ka_src + (col0 >> 6);
        const int off = (lane >> 2) * 512 + 64 * warp + (lane & 3) * 16;
        const bool ok = w.nvalid > 0;
        cp_async16(st_sc + off, ok ? A.nv_scales + tile0 * 512 + off : A.nv_scales, ok ? 16u : 0u);
      }
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
    if (kGather)
      __syncthreads();
    else
      __syncwarp();
    if (kGather) {  // the routed rows' codes: a copy of the staged token codes
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int q = k * 256 + tid;
        const int i = q >> 2, part = q & 3;
        if (i < w.nvalid)
          *reinterpret_cast<uint4 *>(A.nv_codes_out + (w.src_row0 + i) * half_cols + (col0 >> 1) + part * 16) =
              *reinterpret_cast<const uint4 *>(st_codes + i * 64 + part * 16);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = u * 256 + tid;
      const int i = q >> 3, kb = q & 7;
      uint2 raw = make_uint2(0, 0);
      uint32_t sc = 0;
      if (i < w.nvalid) {
        raw = *reinterpret_cast<const uint2 *>(st_codes + i * 64 + kb * 8);
        sc = kGather ? st_sc[i * 8 + kb] : st_sc[(kb >> 2) * 512 + atom_pos(i, kb)];
      }
      if (kGather) s_nvsc[(kb >> 2) * 512 + atom_pos(i, kb)] = (uint8_t)sc;
      store_f16_products<kT8>(s_in, i, kb, raw, sc);
    }
  } else {
    // bf16 -> NVFP4 with the quantizer's block rule (nvfp4_block), codes to
    // global memory, scales to the shared tile; the exact f16 products of the
    // new codes replace the unit's bf16 values in place for phase 2
    __shared__ float s_inv[128];
    __shared__ float s_qt[256];
    const float den6 = __fmul_rn(6.0f, sg);
    // the block-scale table of nvfp4_block_tab applies while every quotient
    // (1 + m / 128) / den6 is a normal fp32 number
    const bool tab = !kRows && !k46 && den6 >= 0x1p-100f && den6 <= 0x1p100f;
    if (!kRows) fill_inv_table(s_inv, sg);
    if (tab) {  // normal mantissas (1 + m / 128), then the subnormal maxima m 2^-133
      const uint32_t t = (uint32_t)tid;
      s_qt[t] = __fdiv_rn(__uint_as_float(t < 128 ? 0x3F800000u | (t << 16) : (t - 128) << 16), den6);
    }
    // every warp reads the tables: one barrier, before any warp has a copy
    // in flight; the tile's rows are then each warp's own (no CTA barrier
    // between a warp's copies landing and its row-wise pass)
    if (!kRows) __syncthreads();
    stage_bf16_tile<kGather, true>(A, w, col0, s_in);
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = u * 256 + tid;
      const int i = q >> 3, kb = q & 7;
      const uint4 *row = reinterpret_cast<const uint4 *>(s_in + i * 256);
      const uint4 va = row[chunk_of(i, 2 * kb)], vb = row[chunk_of(i, 2 * kb + 1)];
      uint2 c;
      uint32_t sc;
      if (kRows) {
        const float sgi = i < w.nvalid ? A.nv_sg_rows[w.src_row0 + i] : 1.0f;
        nvfp4_block(va, vb, sgi, __fmul_rn(6.0f, sgi), c, sc);
      } else if (k46) {
        nvfp4_block46(va, vb, sg, c, sc);
      } else if (tab) {
        nvfp4_block_tab(va, vb, s_qt, s_inv, c, sc);  // an all-zero (padding) block gives scale 0 and zero codes
      } else {
        nvfp4_block(va, vb, sg, den6, c, sc, s_inv);
      }
      if (i < w.nvalid)
        *reinterpret_cast<uint2 *>(A.nv_codes_out + ((w.src_row0 + i) * A.cols + col0 + kb * 16) / 2) = c;
      s_nvsc[(kb >> 2) * 512 + atom_pos(i, kb)] = (uint8_t)sc;
      store_f16_products(s_in, i, kb, c, sc);
    }
  }
  // phase 2 reads every row of the tile: the NVFP4 sources' products written
  // in phase 1, the bf16 source's rows staged per warp
  __syncthreads();

  uint8_t *const out_lane = A.out_codes + out_base + 4 * lane;

  // ---- phase 2 --------------------------------------------------------------
  // warp handles groups of 8 output rows (source columns c8*8 .. c8*8+7);
  // lane handles tokens 4*lane .. 4*lane+3, so tokens 32b .. 32b+31 sit on
  // lanes 8b .. 8b+7.  The lane's two token pairs (4l, 4l+1) and (4l+2, 4l+3)
  // draw from one Philox call each: pair keys (row * cols + column) for the
  // 8 consecutive columns.  Each lane computes the E8M0 scale of one column
  // (lane & 7) of its block and broadcasts its multiplier.
  if constexpr (kT8) {
    // Warp w covers source columns 16w .. 16w + 15: lane 16h + tg owns the
    // column group cg = 2w + h (8 columns) and tokens 8tg .. 8tg + 7, so the
    // 32 tokens of block b sit on lanes 4b .. 4b + 3 of each half-warp.  Each
    // of the lane's token pairs (8tg + 2m, 8tg + 2m + 1) draws the keys of its
    // 8 columns from one Philox call (pair key row * cols + column, as the
    // 4-token pass).  Lane 4b + r ends the block-maximum reduce-scatter with
    // column pair r, computes the E8M0 scales of columns 2r and 2r + 1, and
    // hands their multipliers to the block's four lanes.
    const int tg = lane & 15;
    const int cg = 2 * warp + (lane >> 4);
    const int r = lane & 3;
    uint32_t v[8][4];  // [token j][column pair] exact f16 products
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = 8 * tg + j;
      const uint4 raw = reinterpret_cast<const uint4 *>(s_in + i * 256)[chunk_of8(i, cg)];
      v[j][0] = raw.x; v[j][1] = raw.y; v[j][2] = raw.z; v[j][3] = raw.w;
    }
    uint4 bits[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) bits[m] = make_uint4(0u, 0u, 0u, 0u);
    if (A.sr) {  // rows past the window's data draw too: their values are zeros, which SR keeps
      const uint64_t q = (uint64_t)(((w.src_row0 + 8 * tg) * A.cols + col0 + 8 * cg) >> 3);
      const uint64_t qs = (uint64_t)(A.cols >> 2);  // two rows on (cols % 128 == 0)
#pragma unroll
      for (int m = 0; m < 4; ++m) bits[m] = philox_bits8_rk(q + m * qs, A.off_t, A.rk);
    }
    // column pairs: maxima over the lane's 8 tokens, then a reduce-scatter
    // over the block's 4 lanes that leaves pair r on lane 4b + r
    uint32_t mx[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      uint32_t x = habsmax2(v[0][p], v[1][p]);
#pragma unroll
      for (int j = 2; j < 8; ++j) x = habsmax2(x, v[j][p]);
      mx[p] = x;
    }
    const bool b1 = lane & 2, b0 = lane & 1;
    uint32_t m2p[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t keep = b1 ? mx[q + 2] : mx[q], send = b1 ? mx[q] : mx[q + 2];
      m2p[q] = habsmax2(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 2));
    }
    const uint32_t keep1 = b0 ? m2p[1] : m2p[0], send1 = b0 ? m2p[0] : m2p[1];
    const uint32_t mp = habsmax2(keep1, __shfl_xor_sync(0xFFFFFFFFu, send1, 1));
    float m2a, m2b;  // multipliers of columns 2r and 2r + 1 of the group
    {
      // max_i fp32(p_i * sg) = fp32(max_i p_i * sg): rounding is monotonic
      const float aa = __fmul_rn(fabsf(f16_lo(mp)), sg), ab = __fmul_rn(fabsf(f16_hi(mp)), sg);
      float ma, mb;
      const uint32_t sca = e8m0_scale(aa, &ma), scb = e8m0_scale(ab, &mb);
      // an all-zero block keeps its signed zeros: multiplier 0, not sg * 2^127
      m2a = aa == 0.0f ? 0.0f : __fmul_rn(sg, ma);
      m2b = ab == 0.0f ? 0.0f : __fmul_rn(sg, mb);
      const int c0 = 8 * cg + 2 * r, blk = tg >> 2;
      s_tsc[atom_pos(c0, blk)] = (uint8_t)sca;
      s_tsc[atom_pos(c0 + 1, blk)] = (uint8_t)scb;
    }
    // output rows 8cg .. 8cg + 7, the lane's 8 tokens each (a half-warp
    // writes one whole 128-byte row per store)
    uint8_t *out8 = A.out_codes + out_base + 8 * tg + (int64_t)(8 * cg) * out_stride;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int p = k >> 1, h = k & 1;
      const float m2 = __shfl_sync(0xFFFFFFFFu, h ? m2b : m2a, p, 4);  // from lane 4 * (lane / 4) + p
      float x[8];
#pragma unroll
      for (int j = 0; j < 8; j += 2)
        mul2_rn(h ? f16_hi(v[j][p]) : f16_lo(v[j][p]), h ? f16_hi(v[j + 1][p]) : f16_lo(v[j + 1][p]), m2, x[j],
                x[j + 1]);
      uint32_t lo, hi;
      if (A.sr) {
        // tokens 2m, 2m + 1 take half h of word p of pair m's draws (U, then bitrev16(U))
        const uint32_t sel = h ? 0x7632u : 0x5410u;
        const uint32_t u0 = __byte_perm(word_of(bits[0], p), word_of(bits[1], p), sel);
        const uint32_t u1 = __byte_perm(word_of(bits[2], p), word_of(bits[3], p), sel);
        lo = cvt_e4m3x4_sr(x[0], x[1], x[2], x[3], ~u0);
        hi = cvt_e4m3x4_sr(x[4], x[5], x[6], x[7], ~u1);
      } else {
        lo = cvt_e4m3x2_rn(x[0], x[1]) | (cvt_e4m3x2_rn(x[2], x[3]) << 16);
        hi = cvt_e4m3x2_rn(x[4], x[5]) | (cvt_e4m3x2_rn(x[6], x[7]) << 16);
      }
      *reinterpret_cast<uint2 *>(out8) = make_uint2(lo, hi);
      out8 += out_stride;
    }
  } else {
  float sg_tok[4];  // per-token outer scales of this lane's tokens (kRows)
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = 4 * lane + j;
    sg_tok[j] = (kRows && i < w.nvalid) ? A.nv_sg_rows[w.src_row0 + i] : 0.0f;
  }
  // Philox counters: pair keys (row * cols + column) / 8 of token 4l's columns
  // c8 * 8 .. c8 * 8 + 7 are q0 + c8, token 4l + 2's are q0 + c8 + cols / 4
  // (cols and col0 are multiples of 128)
  const uint64_t q0 = (uint64_t)(((w.src_row0 + 4 * lane) * A.cols + col0) >> 3);
  const uint64_t q2 = (uint64_t)(A.cols >> 2);
#pragma unroll 1
  for (int c8 = warp; c8 < 16; c8 += 8) {
    uint32_t v[4][4];  // [token j][column pair] packed 16-bit values
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = 4 * lane + j;
      const uint4 raw = reinterpret_cast<const uint4 *>(s_in + i * 256)[chunk_of(i, c8)];
      v[j][0] = raw.x; v[j][1] = raw.y; v[j][2] = raw.z; v[j][3] = raw.w;
    }
    uint4 ba = make_uint4(0, 0, 0, 0), bb = make_uint4(0, 0, 0, 0);
    if (A.sr) {  // rows past the window's data draw too: their values are zeros, which SR keeps
      ba = philox_bits8_rk(q0 + c8, A.off_t, A.rk);
      bb = philox_bits8_rk(q0 + c8 + q2, A.off_t, A.rk);
    }
    if constexpr (kRows) {
      // per-token outer scales: the dequantized values fp32(p * sg_token)
      // first, their block maximum by a reduce-scatter over the 8 lanes of a
      // block (lane & 7 ends with its own column), then SR of fp32(x * 2^-s)
      float xv[4][8];
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          xv[j][2 * q] = __fmul_rn(f16_lo(v[j][q]), sg_tok[j]);
          xv[j][2 * q + 1] = __fmul_rn(f16_hi(v[j][q]), sg_tok[j]);
        }
      float mk[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mk[k] = fmaxf(fmaxf(fabsf(xv[0][k]), fabsf(xv[1][k])), fmaxf(fabsf(xv[2][k]), fabsf(xv[3][k])));
      const bool b2 = lane & 4, b1 = lane & 2, b0 = lane & 1;
      float k4[4], k2[2];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float send = b2 ? mk[k] : mk[k + 4];
        k4[k] = fmaxf(b2 ? mk[k + 4] : mk[k], __shfl_xor_sync(0xFFFFFFFFu, send, 4));
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float send = b1 ? k4[k] : k4[k + 2];
        k2[k] = fmaxf(b1 ? k4[k + 2] : k4[k], __shfl_xor_sync(0xFFFFFFFFu, send, 2));
      }
      const float amax_own = fmaxf(b0 ? k2[1] : k2[0], __shfl_xor_sync(0xFFFFFFFFu, b0 ? k2[0] : k2[1], 1));
      float mult_own;
      const uint32_t sc = e8m0_scale(amax_own, &mult_own);
      s_tsc[atom_pos(c8 * 8 + (lane & 7), lane >> 3)] = (uint8_t)sc;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int c = c8 * 8 + k;
        const float m2 = __shfl_sync(0xFFFFFFFFu, mult_own, k, 8);  // from lane 8 * (lane / 8) + k
        const int p = k >> 1, h = k & 1;
        float x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = __fmul_rn(xv[j][k], m2);
        uint32_t packed;
        if (A.sr) {
          const uint32_t wa = p == 0 ? ba.x : p == 1 ? ba.y : p == 2 ? ba.z : ba.w;
          const uint32_t wb = p == 0 ? bb.x : p == 1 ? bb.y : p == 2 ? bb.z : bb.w;
          const uint32_t u = __byte_perm(wa, wb, h ? 0x7632 : 0x5410);
          packed = cvt_e4m3x4_sr(x[0], x[1], x[2], x[3], ~u);
        } else {
          packed = cvt_e4m3x2_rn(x[0], x[1]) | (cvt_e4m3x2_rn(x[2], x[3]) << 16);
        }
        *reinterpret_cast<uint32_t *>(out_lane + (int64_t)c * out_stride) = packed;
      }
      continue;
    }
    // column pairs (2p, 2p+1): maxima over the lane's 4 tokens, then over the
    // 8 lanes of the block by a reduce-scatter (keep half, send half), after
    // which lanes 2q and 2q+1 of a block both hold pair q over all 32 tokens:
    // the pair of the lane's own column k_own = lane & 7
    uint32_t m[4];
#pragma unroll
    for (int p = 0; p < 4; ++p)
      m[p] = kNvfp4 ? habsmax2(habsmax2(v[0][p], v[1][p]), habsmax2(v[2][p], v[3][p]))
                    : bf16x2_absmax(bf16x2_absmax(v[0][p], v[1][p]), bf16x2_absmax(v[2][p], v[3][p]));
    const bool b2 = lane & 4, b1 = lane & 2;
    uint32_t m4[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t keep = b2 ? m[q + 2] : m[q], send = b2 ? m[q] : m[q + 2];
      const uint32_t got = __shfl_xor_sync(0xFFFFFFFFu, send, 4);
      m4[q] = kNvfp4 ? habsmax2(keep, got) : bf16x2_absmax(keep, got);
    }
    uint32_t mp;
    {
      const uint32_t keep = b1 ? m4[1] : m4[0], send = b1 ? m4[0] : m4[1];
      const uint32_t got = __shfl_xor_sync(0xFFFFFFFFu, send, 2);
      mp = kNvfp4 ? habsmax2(keep, got) : bf16x2_absmax(keep, got);
      const uint32_t got1 = __shfl_xor_sync(0xFFFFFFFFu, mp, 1);
      mp = kNvfp4 ? habsmax2(mp, got1) : bf16x2_absmax(mp, got1);
    }
    // this lane's column: k_own = lane & 7
    float m2_own;
    {
      const int k_own = lane & 7;
      float amax, mult;
      if (kNvfp4) {
        // max_i fp32(p_i * sg) = fp32(max_i p_i * sg): rounding is monotonic
        amax = __fmul_rn(fabsf((k_own & 1) ? f16_hi(mp) : f16_lo(mp)), sg);
      } else {
        amax = fabsf((k_own & 1) ? bf16_hi(mp) : bf16_lo(mp));
      }
      const uint32_t sc = e8m0_scale(amax, &mult);
      // NVFP4: fp32(fp32(p * sg) * 2^-s) == fp32(p * (sg * 2^-s)) for the
      // normal-range values the contract covers (the power of two is exact);
      // an all-zero block keeps its signed zeros: multiplier 0, not sg * 2^127
      m2_own = kNvfp4 ? (amax == 0.0f ? 0.0f : __fmul_rn(sg, mult)) : mult;
      s_tsc[atom_pos(c8 * 8 + k_own, lane >> 3)] = (uint8_t)sc;
    }
    // output rows c8 * 8 .. c8 * 8 + 7, one stepped pointer
    uint8_t *out_row = out_lane + (int64_t)(c8 * 8) * out_stride;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float m2 = __shfl_sync(0xFFFFFFFFu, m2_own, k, 8);  // from lane 8 * (lane / 8) + k
      const int p = k >> 1, h = k & 1;
      float x[4];
      if (kNvfp4) {
#pragma unroll
        for (int j = 0; j < 4; j += 2)
          mul2_rn(h ? f16_hi(v[j][p]) : f16_lo(v[j][p]), h ? f16_hi(v[j + 1][p]) : f16_lo(v[j + 1][p]), m2, x[j],
                  x[j + 1]);
      } else {  // m2 is a power of two: one mixed-precision FMA per value
        const uint16_t mb = pow2_bf16_bits(m2);
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = h ? bf16_hi_times(v[j][p], mb) : bf16_lo_times(v[j][p], mb);
      }
      uint32_t packed;
      if (A.sr) {
        const uint32_t wa = p == 0 ? ba.x : p == 1 ? ba.y : p == 2 ? ba.z : ba.w;
        const uint32_t wb = p == 0 ? bb.x : p == 1 ? bb.y : p == 2 ? bb.z : bb.w;
        // Ua = half h of wa (tokens 4l, 4l+1), Ub = half h of wb (tokens 4l+2, 4l+3)
        const uint32_t u = __byte_perm(wa, wb, h ? 0x7632 : 0x5410);
        packed = cvt_e4m3x4_sr(x[0], x[1], x[2], x[3], ~u);
      } else {
        packed = cvt_e4m3x2_rn(x[0], x[1]) | (cvt_e4m3x2_rn(x[2], x[3]) << 16);
      }
      *reinterpret_cast<uint32_t *>(out_row) = packed;
      out_row += out_stride;
    }
  }
  }
  __syncthreads();

  // ---- phase 3 --------------------------------------------------------------
  if (tid < 32) {
    reinterpret_cast<uint4 *>(A.out_scales + tile_idx * 512)[tid] = reinterpret_cast<const uint4 *>(s_tsc)[tid];
  } else if (tid < 64 && A.row_codes != nullptr) {  // zero tiles for padding windows too
    reinterpret_cast<uint4 *>(A.row_scales + ((w.rp0 >> 7) * A.row_ka + (col0 >> 7)) * 512)[tid - 32] =
        reinterpret_cast<const uint4 *>(s_rsc)[tid - 32];
  } else if (kNvOut && tid >= 64 && tid < 128) {  // the two NVFP4 tiles (zeros for padding)
    reinterpret_cast<uint4 *>(A.nv_scales_out + ((w.rp0 >> 7) * A.nv_ka + (col0 >> 6)) * 512)[tid - 64] =
        reinterpret_cast<const uint4 *>(s_nvsc)[tid - 64];
  }
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
static int launch_status(cudaError_t e) { return e == cudaSuccess ? NV_OK : NV_ERR_CUDA; }

int launch_amax(const uint16_t *x, int64_t batch, int64_t per_batch, float *partial, int nblk, float *sg_out,
                cudaStream_t s) {
  amax_partial_kernel<<<dim3(nblk, (unsigned)batch), 256, 0, s>>>(x, per_batch, partial, nblk);
  outer_scale_finalize_kernel<<<(unsigned)batch, 32, 0, s>>>(partial, nblk, sg_out);
  return launch_status(cudaGetLastError());
}

// the amax pass of the gathered rows x[row_src[r]]: row_amax holds src_rows
// floats when src_rows <= rows
int launch_amax_gather(const uint16_t *x, const int32_t *row_src, int64_t src_rows, int64_t rows, int64_t cols,
                       float *partial, int nblk, float *row_amax, float *sg_out, int *status, cudaStream_t s) {
  if (src_rows <= rows) {  // the tokens once each, then the maximum over the row map
    if (src_rows > 0) token_amax_kernel<<<(unsigned)((src_rows + 7) / 8), 256, 0, s>>>(x, src_rows, cols, row_amax);
    gather_amax_partial_kernel<<<nblk, 256, 0, s>>>(row_amax, row_src, src_rows, rows, partial, nblk, status);
  } else {  // more tokens than rows: read the routed rows themselves
    amax_gather_partial_kernel<<<nblk, 256, 0, s>>>(x, row_src, src_rows, rows, cols, partial, nblk, status);
  }
  outer_scale_finalize_kernel<<<1, 32, 0, s>>>(partial, nblk, sg_out);
  return launch_status(cudaGetLastError());
}

// sg = amax / 2688 (1 for a zero amax) in place, exactly as the amax pass
// finishes (one partial maximum)
int launch_outer_scale_from_amax(float *amax_in_sg_out, cudaStream_t s) {
  outer_scale_finalize_kernel<<<1, 32, 0, s>>>(amax_in_sg_out, 1, amax_in_sg_out);
  return launch_status(cudaGetLastError());
}

__global__ void __launch_bounds__(256) row_outer_scale_from_amax_kernel(float *__restrict__ buf, int64_t n) {
  const int64_t r = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (r >= n) return;
  const float a = buf[r];
  buf[r] = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 2688.0f);
}

int launch_row_outer_scale_from_amax(float *amax_in_sg_out, int64_t n, cudaStream_t s) {
  if (n == 0) return NV_OK;
  row_outer_scale_from_amax_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(amax_in_sg_out, n);
  return launch_status(cudaGetLastError());
}

int launch_row_outer_scale(const uint16_t *x, int64_t rows, int64_t cols, float *sg_rows, cudaStream_t s) {
  if (rows == 0) return NV_OK;
  row_outer_scale_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(x, rows, cols, sg_rows);
  return launch_status(cudaGetLastError());
}

int launch_nvfp4_quant(const uint16_t *x, int64_t batch, int64_t rows, int64_t cols, const int32_t *groups, int E,
                       const float *sg, uint8_t *codes, uint8_t *scales, int *status, cudaStream_t s,
                       const float *sg_rows, int four_six) {
  NvQuantArgs A;
  A.x = x; A.rows = rows; A.cols = cols; A.groups = groups; A.E = E;
  A.wpb = (int)((rows + 127) / 128);
  A.sg = sg; A.sg_rows = sg_rows; A.four_six = four_six;
  A.codes = codes; A.scales = scales; A.ka = (cols / 16 + 3) / 4; A.status = status;
  const int64_t nwin = groups ? nvfp4moe_padded_cap(rows, E) / 128 : batch * A.wpb;
  const int64_t nchunk = (cols / 16 + 15) / 16;
  if (nwin == 0) return NV_OK;
  nvfp4_quant_kernel<<<dim3((unsigned)nchunk, (unsigned)nwin), 256, 0, s>>>(A);
  return launch_status(cudaGetLastError());
}

int launch_mxfp8_rowwise(const uint16_t *x, int64_t rows, int64_t cols, const int32_t *groups, int E, int sr,
                         uint64_t seed, uint64_t off, uint8_t *codes, uint8_t *scales, int *status, cudaStream_t s) {
  MxRowArgs A;
  A.x = x; A.rows = rows; A.cols = cols; A.groups = groups; A.E = E; A.sr = sr; A.seed = seed; A.offset = off;
  A.rk = philox_round_keys(seed);
  A.codes = codes; A.scales = scales; A.ka = (cols / 32 + 3) / 4; A.status = status;
  const int64_t P = groups ? nvfp4moe_padded_cap(rows, E) : ((rows + 127) / 128) * 128;
  const int64_t nwin = P / 128, nchunk = (cols / 32 + 7) / 8;
  if (nwin == 0) return NV_OK;
  mxfp8_rowwise_kernel<<<dim3((unsigned)nchunk, (unsigned)nwin), 256, 0, s>>>(A);
  return launch_status(cudaGetLastError());
}

static size_t mx_t_smem(bool nvfp4_source) { return (nvfp4_source ? kNvStage : 0) + (size_t)kTileSmem; }

int launch_mx_transpose_bf16(const uint16_t *x, int64_t rows, int64_t cols, const int32_t *groups, int E, int sr,
                             uint64_t seed, uint64_t off_t, uint64_t off_row, uint8_t *codes_t, uint8_t *scales_t,
                             uint8_t *codes_row, uint8_t *scales_row, int *status, cudaStream_t s) {
  MxTArgs A = {};
  A.x = x; A.rows = rows; A.cols = cols; A.groups = groups; A.E = E; A.grouped = 1; A.sr = sr;
  A.seed = seed; A.off_t = off_t; A.off_row = off_row;
  A.rk = philox_round_keys(seed);
  const int64_t P = groups ? nvfp4moe_padded_cap(rows, E) : ((rows + 127) / 128) * 128;
  A.out_codes = codes_t; A.out_scales = scales_t; A.out_stride = P; A.out_ka = P / 128;
  A.row_codes = codes_row; A.row_scales = scales_row; A.row_ka = cols / 128;
  A.status = status;
  const size_t sm = mx_t_smem(false);
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(mx_transpose_kernel<kSrcBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    attr_set = true;
  }
  if (P == 0) return NV_OK;
  mx_transpose_kernel<kSrcBf16><<<dim3((unsigned)(cols / 128), (unsigned)(P / 128)), 256, sm, s>>>(A);
  return launch_status(cudaGetLastError());
}

int launch_requant(const uint8_t *codes, const uint8_t *scales, const float *sg, int64_t batch, int64_t rows,
                   int64_t cols, const int32_t *groups, int E, uint64_t seed, uint64_t off, uint8_t *out_codes,
                   uint8_t *out_scales, int *status, cudaStream_t s, const float *sg_rows) {
  MxTArgs A = {};
  A.nv_codes = codes; A.nv_scales = scales; A.nv_sg = sg; A.nv_sg_rows = sg_rows; A.rows = rows; A.cols = cols; A.groups = groups; A.E = E;
  A.sr = 1; A.seed = seed; A.off_t = off; A.status = status;
  A.rk = philox_round_keys(seed);
  A.out_codes = out_codes; A.out_scales = out_scales;
  int64_t nwin;
  if (groups) {
    const int64_t P = nvfp4moe_padded_cap(rows, E);
    A.grouped = 1; A.out_stride = P; A.out_ka = P / 128; nwin = P / 128;
  } else {
    A.grouped = 0; A.wpb = (int)(rows / 128); A.out_ka = rows / 128; nwin = batch * A.wpb;
  }
  const size_t sm = mx_t_smem(true);
  auto k = sg_rows ? mx_transpose_kernel<kSrcNvfp4, true> : mx_transpose_kernel<kSrcNvfp4, false>;
  static bool attr_set[2] = {false, false};
  if (!attr_set[sg_rows ? 1 : 0]) {
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    attr_set[sg_rows ? 1 : 0] = true;
  }
  if (nwin == 0) return NV_OK;
  k<<<dim3((unsigned)(cols / 128), (unsigned)nwin), 256, sm, s>>>(A);
  return launch_status(cudaGetLastError());
}

// the gathered re-quantization: routed row r of the grouped output is token
// row row_src[r] of the NVFP4 token matrix (codes [src_rows][cols / 2],
// batched scale layout); its codes and scales are copied to the routed
// layout and its values re-quantized (transposed MXFP8 SR)
int launch_requant_gather(const uint8_t *tok_codes, const uint8_t *tok_scales, const float *sg,
                          const int32_t *row_src, int64_t src_rows, int64_t rows, int64_t cols,
                          const int32_t *groups, int E, uint8_t *codes, uint8_t *scales, uint64_t seed, uint64_t off,
                          uint8_t *out_codes, uint8_t *out_scales, int *status, cudaStream_t s) {
  MxTArgs A = {};
  A.nv_codes = tok_codes; A.nv_scales = tok_scales; A.nv_sg = sg; A.row_src = row_src; A.src_rows = src_rows;
  A.rows = rows; A.cols = cols; A.groups = groups; A.E = E;
  A.nv_codes_out = codes; A.nv_scales_out = scales; A.nv_ka = cols / 64;
  A.sr = 1; A.seed = seed; A.off_t = off; A.status = status;
  A.rk = philox_round_keys(seed);
  A.out_codes = out_codes; A.out_scales = out_scales;
  const int64_t P = nvfp4moe_padded_cap(rows, E);
  A.grouped = 1; A.out_stride = P; A.out_ka = P / 128;
  const size_t sm = mx_t_smem(true);
  auto k = mx_transpose_kernel<kSrcNvfp4, false, false, true>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    attr_set = true;
  }
  if (P == 0) return NV_OK;
  k<<<dim3((unsigned)(cols / 128), (unsigned)(P / 128)), 256, sm, s>>>(A);
  return launch_status(cudaGetLastError());
}

int launch_nvfp4_requant(const uint16_t *x, const float *sg, int64_t batch, int64_t rows, int64_t cols,
                         const int32_t *groups, int E, uint8_t *codes, uint8_t *scales, uint64_t seed, uint64_t off,
                         uint8_t *out_codes, uint8_t *out_scales, int *status, cudaStream_t s, const float *sg_rows,
                         int four_six, const int32_t *row_src, int64_t src_rows) {
  MxTArgs A = {};
  A.x = x; A.row_src = row_src; A.src_rows = src_rows; A.nv_sg = sg; A.nv_sg_rows = sg_rows; A.rows = rows; A.cols = cols; A.groups = groups; A.E = E;
  A.nv_codes_out = codes; A.nv_scales_out = scales; A.nv_ka = cols / 64;
  A.sr = 1; A.seed = seed; A.off_t = off; A.status = status;
  A.rk = philox_round_keys(seed);
  A.out_codes = out_codes; A.out_scales = out_scales;
  int64_t nwin;
  if (groups) {
    const int64_t P = nvfp4moe_padded_cap(rows, E);
    A.grouped = 1; A.out_stride = P; A.out_ka = P / 128; nwin = P / 128;
  } else {
    A.grouped = 0; A.wpb = (int)(rows / 128); A.out_ka = rows / 128; nwin = batch * A.wpb;
  }
  const size_t sm = mx_t_smem(false);
  if (row_src && (sg_rows || four_six)) return NV_ERR_ARG;  // gathered rows: per-tensor scale, plain rule
  const int which = sg_rows ? 1 : four_six ? 2 : row_src ? 3 : 0;
  auto k = which == 1   ? mx_transpose_kernel<kSrcBf16ToNvfp4, true>
           : which == 2 ? mx_transpose_kernel<kSrcBf16ToNvfp4, false, true>
           : which == 3 ? mx_transpose_kernel<kSrcBf16ToNvfp4, false, false, true>
                        : mx_transpose_kernel<kSrcBf16ToNvfp4, false>;
  static bool attr_set[4] = {false, false, false, false};
  if (!attr_set[which]) {
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    attr_set[which] = true;
  }
  if (nwin == 0) return NV_OK;
  k<<<dim3((unsigned)(cols / 128), (unsigned)nwin), 256, sm, s>>>(A);
  return launch_status(cudaGetLastError());
}

}  // namespace nvm
