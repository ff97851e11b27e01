// Grouped block-scaled expert GEMMs on the 5th-generation tensor cores
// (tcgen05), the three expert GEMMs of the layer's training step:
//   NVFP4 forward   y_e  = x_q,e w_q,e^T      kind::mxf4nvf4, E4M3 scales / 16
//   MXFP8 dgrad     dx_e = g_e w_e            kind::mxf8f6f4, E8M0 scales / 32
//   MXFP8 wgrad     dw_e = g_e^T x_q,e        kind::mxf8f6f4, contraction over
//                                             the expert's padded tokens
// "End-to-End 4-Bit Training", "Block-scaled backward passes": a block-scaled
// dot product multiplies pairs of a 16- (or 32-) value block from each operand,
// sums them and scales the sum by both block scales; "Kernels for
// low-precision training": the MoE layer is dominated by these GEMMs.
//
// Persistent kernel looping over 128 x 128 output tiles in a static
// round-robin order.  Default: two CTAs per SM, each with a 3-stage ring and
// one accumulator, so one CTA's epilogue and barrier waits are covered by the
// other CTA's MMAs (measured faster than one CTA per SM with a 6-stage ring
// and two accumulators, which NVFP4MOE_GEMM_VARIANT=1 selects).  Roles:
//   warp 0      TMA producer: A/B tiles (128-byte swizzle) and whole 512-byte
//               128x4 scale tiles (1-D bulk copies) into a STAGES-deep ring,
//               continuously across tiles
//   warp 1      allocates tensor memory; one thread copies each stage's scales
//               to tensor memory (tcgen05.cp, one buffer per ring stage) and
//               issues 4 block-scaled MMAs per stage into the fp32
//               accumulator (or alternates two, variant 1)
//   warps 2-5   epilogue: tcgen05.ld of the finished accumulator into
//               registers, release of the accumulator, then outer-scale
//               multiply and 32-byte streaming stores of the rows that belong
//               to the expert
// Every wait is bounded: a wait that runs out records NV_ERR_TIMEOUT and
// raises a CTA-wide abort flag so that the other roles stop too; the producer
// waits (bounded) for its own copies and tensor memory is always freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "launch.h"
#include "rht_s2f6_block.cuh"

namespace nvm {

// ---------------------------------------------------------------------------
// PTX wrappers (tcgen05, TMA, bulk copies)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// 8-byte asynchronous global -> shared copies in commit groups
__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev_group() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all_groups() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void mma_nvf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
// The same with the block16 scale form (one E4M3 scale per 16 values, any
// K): with the instruction descriptor's K-dimension bit (bit 31) set this is
// the K = 96 form of sm_103a, which does 1.5x the work of K = 64 in the same
// issue time.  Its six scales per row are consecutive bytes of the 128x4
// scale layout starting at byte `id` (descriptor bits 29-30 for A, 4-5 for
// B) of the given scale column, continuing in the next 4-column atom.
__device__ __forceinline__ void mma_nvf4_b16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                             uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.block16 [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
constexpr uint32_t kIdescK96 = 1u << 31;
__host__ __device__ constexpr uint32_t idesc_sf_id(uint32_t id) { return (id << 29) | (id << 4); }

__device__ __forceinline__ void mma_mxf8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
// 32 consecutive accumulator columns of this warp's 32 lanes, no wait
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t *v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor, K-major operand tile with rows of 128 bytes
// in the 128-byte swizzle (8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Descriptor of one 512-byte scale tile: 32 rows of 16 bytes, no swizzle.
__device__ __forceinline__ uint64_t desc_sf(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}

// ---------------------------------------------------------------------------
// configuration
// ---------------------------------------------------------------------------
constexpr int cpow2(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

constexpr int kBN = 128;  // output tile columns (and rows: 128)

template <int KIND, int STAGES, int NACC>
struct Cfg {
  static constexpr bool kFp4 = KIND == kGemmNvfp4Fwd || KIND == kGemmNvfp4FwdSwiglu;
  static constexpr int kAtomsPerStage = kFp4 ? 4 : 1;  // 128x4 scale tiles per 128 rows per stage
  static constexpr int A_BYTES = 128 * 128;
  static constexpr int B_BYTES = kBN * 128;
  static constexpr int SFA_BYTES = kAtomsPerStage * 512;
  static constexpr int SFB_BYTES = (kBN / 128) * SFA_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int SFA_COLS = kAtomsPerStage * 4;  // tensor-memory columns per stage
  static constexpr int SFB_COLS = kAtomsPerStage * (kBN / 32);
  static constexpr int SF_COLS = SFA_COLS + SFB_COLS;
  static constexpr int ACC_COLS = NACC * kBN;           // one or two accumulators
  // one scale buffer per ring stage: a stage's buffer is rewritten only after
  // the producer has refilled that stage, i.e. after its previous MMAs retired
  static constexpr int TMEM_COLS = cpow2(ACC_COLS + STAGES * SF_COLS);
  static constexpr int NBARS = 2 * STAGES + 2 * NACC + 1;  // full, empty, acc_full[], acc_empty[], mma_done
  static constexpr uint32_t IDESC =
      (kFp4 ? ((1u << 7) | (1u << 10)) : (1u << 23)) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  static size_t smem_bytes(int E) {
    return 1024 + (size_t)STAGES * STAGE_BYTES + NBARS * 8 + 32 + (size_t)(E + 1) * 8 + 64;
  }
  static_assert(TMEM_COLS <= 512, "tensor memory");
};

struct GemmArgs {
  const uint8_t *a_scales, *b_scales;
  const float *a_sg, *b_sg;
  const int32_t *groups;
  int E;
  int64_t M_total, N, K;
  int ntn;       // output column tiles
  int ntm;       // wgrad: output row tiles per expert
  int64_t ka;    // scale tiles per 128 rows (A and B)
  void *out;
  int out_fp32;
  int64_t out_ld;
  int *status;
  uint64_t wait_limit;
  // kGemmNvfp4FwdSwiglu
  void *h;
  unsigned *h_amax;
  int64_t I;
  int a_sg_rows;   // a_sg is per row of A (per token)
  int h_amax_rows;  // h_amax is per row of h
  // NVFP4 forward: RHT-32 + S2F6 of the bf16 output rows (null: none)
  int8_t *s2f6_codes;
  uint8_t *s2f6_scales;
  RhtSigns rht;
  // kGemmMxfp8Dx: the SwiGLU backward of the bf16 output dh (the K output
  // columns) with y13 [M_total][2K] bf16; `out` is then dy13 [M_total][2K]
  const uint16_t *swb_y13;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Stores 128 bytes of each of a warp's 32 output rows (lane = row; w[] =
// the lane's 32 words, row rr at seg0 + rr * ld_bytes) as whole 128-byte
// lines.  Each group of four lanes transposes its 4 x 4 block of 32-byte
// chunks with two butterfly exchanges (over lane bits 1 and 0), after which
// lane 4g + i holds chunk i of rows 4g .. 4g + 3; store k then writes row
// 4g + k's 128 bytes with the group's four lanes: eight full lines per
// instruction, where storing each lane's own row touches 32 lines.  Rows from
// `nrows` on are not stored.  Every lane of the warp must call it.
__device__ __forceinline__ void store_segment_coalesced(uint8_t *seg0, int64_t ld_bytes, uint32_t (&w)[32], int lane,
                                                        int nrows) {
  const int g = lane >> 2, i = lane & 3;
#pragma unroll
  for (int d = 2; d >= 1; d >>= 1) {
    const bool b = (lane & d) != 0;
#pragma unroll
    for (int j0 = 0; j0 < 4; ++j0) {
      if (j0 & d) continue;
      const int j1 = j0 | d;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t got = __shfl_xor_sync(0xFFFFFFFFu, b ? w[8 * j0 + e] : w[8 * j1 + e], d);
        if (b)
          w[8 * j0 + e] = got;
        else
          w[8 * j1 + e] = got;
      }
    }
  }
  uint8_t *p = seg0 + (int64_t)(4 * g) * ld_bytes + 32 * i;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (4 * g + k < nrows)
      st_cs_v8(p, w[8 * k], w[8 * k + 1], w[8 * k + 2], w[8 * k + 3], w[8 * k + 4], w[8 * k + 5], w[8 * k + 6],
               w[8 * k + 7]);
    p += ld_bytes;
  }
}

// SwiGLU epilogue of one accumulator row segment: r[0..63] the gate and
// r[64..127] the up columns of hidden features col0 .. col0 + 63 of output row
// `orow`.  y13 = bf16(acc * alpha) exactly as the plain bf16 output; h from
// the rounded gate and up with the SwiGLU kernel's arithmetic; max |h| of the
// rows that exist, one atomic per warp, or per row with per-token scales (max
// is order-free).  Every lane of the warp must call it.
__device__ __forceinline__ void swiglu_epilogue(const GemmArgs &A, const uint32_t *r, float alpha, bool store,
                                                int64_t orow, int64_t col0, int lane) {
  float hmax = 0.0f;
  if (store) {
    uint16_t *yg = static_cast<uint16_t *>(A.out) + orow * (2 * A.I) + col0;
    uint16_t *yu = yg + A.I;
    uint16_t *hp = static_cast<uint16_t *>(A.h) + orow * A.I + col0;
#pragma unroll
    for (int i = 0; i < 64; i += 16) {
      uint32_t wg[8], wu[8], wh[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        wg[k] = pack_bf16x2(__fmul_rn(__uint_as_float(r[i + 2 * k]), alpha),
                            __fmul_rn(__uint_as_float(r[i + 2 * k + 1]), alpha));
        wu[k] = pack_bf16x2(__fmul_rn(__uint_as_float(r[64 + i + 2 * k]), alpha),
                            __fmul_rn(__uint_as_float(r[64 + i + 2 * k + 1]), alpha));
        const float h0 = swiglu_h(bf16_lo(wg[k]), bf16_lo(wu[k]));
        const float h1 = swiglu_h(bf16_hi(wg[k]), bf16_hi(wu[k]));
        wh[k] = f32_to_bf16_bits(h0) | (f32_to_bf16_bits(h1) << 16);
        hmax = fmaxf(hmax, fmaxf(fabsf(bf16_lo(wh[k])), fabsf(bf16_hi(wh[k]))));
      }
      st_cs_v8(yg + i, wg[0], wg[1], wg[2], wg[3], wg[4], wg[5], wg[6], wg[7]);
      st_cs_v8(yu + i, wu[0], wu[1], wu[2], wu[3], wu[4], wu[5], wu[6], wu[7]);
      st_cs_v8(hp + i, wh[0], wh[1], wh[2], wh[3], wh[4], wh[5], wh[6], wh[7]);
    }
  }
  if (A.h_amax_rows) {  // per token: this thread's row
    if (store && hmax > 0.0f) atomicMax(A.h_amax + orow, __float_as_uint(hmax));
  } else {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) hmax = fmaxf(hmax, __shfl_xor_sync(0xFFFFFFFFu, hmax, d));
    if (lane == 0 && hmax > 0.0f) atomicMax(A.h_amax, __float_as_uint(hmax));
  }
}

// The y13 lines (gate and up, NC columns from col0) that swiglu_bwd_epilogue
// will read for row orow, fetched into L2 while the tile's MMAs run (the
// epilogue warps are idle until its accumulator is complete).
template <int NC>
__device__ __forceinline__ void prefetch_swiglu_rows(const GemmArgs &A, int64_t orow, int64_t col0) {
  const uint16_t *yg = A.swb_y13 + orow * (2 * A.K) + col0;
#pragma unroll
  for (int i = 0; i < NC; i += 64) {  // 128-byte lines
    asm volatile("prefetch.global.L2 [%0];" ::"l"(yg + i));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(yg + A.K + i));
  }
}

// SwiGLU backward epilogue of a warp's 32 output rows of the dgrad GEMM dh =
// g2 w2 (lane = row; r[0..NC) the lane's fp32 dh of columns col0 .. col0 +
// NC; rows from `nrows` on do not exist).  Each dh is rounded to bf16 exactly
// as the plain bf16 output (alpha is 1) and combined with the row's gate and
// up values of y13 by the SwiGLU backward kernel's arithmetic: dgate to
// dy13 columns col0 .., dup to I + col0 .. (I = K).  Per 64 columns, the
// packed dh rows go through the 4 x 4 chunk transpose of
// store_segment_coalesced, after which lane 4g + i holds 16 columns (chunk i)
// of rows 4g .. 4g + 3: the y13 loads and dy13 stores then cover whole
// 128-byte lines (eight per warp instruction) instead of 32 lines of 16 or 32
// bytes.  y13, dy13 and their row length 32-byte aligned.  Every lane of the
// warp must call it.
template <int NC>
__device__ __forceinline__ void swiglu_bwd_epilogue(const GemmArgs &A, const uint32_t *r, int64_t row0,
                                                    int64_t col0, int lane, int nrows) {
  static_assert(NC % 64 == 0, "64-column segments");
  const int64_t I = A.K, ld = 2 * I;
  const int g = lane >> 2, ci = lane & 3;
  // every segment's dh packed first (the fp32 values are then dead), so that
  // a segment's y13 loads can all be in flight while its dh is transposed
  uint32_t w[NC / 64][32];
#pragma unroll
  for (int S = 0; S < NC / 64; ++S)
#pragma unroll
    for (int k = 0; k < 32; ++k)
      w[S][k] = pack_bf16x2(__uint_as_float(r[64 * S + 2 * k]), __uint_as_float(r[64 * S + 2 * k + 1]));
#pragma unroll
  for (int S = 0; S < NC / 64; ++S) {
    // after the transpose lane 4g + ci holds columns col0 + 64 S + 16 ci ..
    // + 15 of rows 4g .. 4g + 3: their gate and up, 32 bytes each, two rows'
    // worth in flight at a time (the first pair's during the transpose)
    const int64_t c = col0 + 64 * S + 16 * ci;
#pragma unroll
    for (int kb = 0; kb < 4; kb += 2) {
      uint32_t gl[2][8], ul[2][8];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (4 * g + kb + k < nrows) {
          const uint16_t *yg = A.swb_y13 + (row0 + 4 * g + kb + k) * ld + c;
          ld_stream_v8(yg, gl[k]);
          ld_stream_v8(yg + I, ul[k]);
        }
      }
      if (kb == 0) {
#pragma unroll
        for (int d = 2; d >= 1; d >>= 1) {
          const bool b = (lane & d) != 0;
#pragma unroll
          for (int j0 = 0; j0 < 4; ++j0) {
            if (j0 & d) continue;
            const int j1 = j0 | d;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const uint32_t got = __shfl_xor_sync(0xFFFFFFFFu, b ? w[S][8 * j0 + e] : w[S][8 * j1 + e], d);
              if (b)
                w[S][8 * j0 + e] = got;
              else
                w[S][8 * j1 + e] = got;
            }
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (4 * g + kb + k >= nrows) continue;
        uint32_t wg[8], wu[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t dw = w[S][8 * (kb + k) + e];
          float a0, b0, a1, b1;
          swiglu_bwd_f32x2(bf16_lo(dw), bf16_hi(dw), bf16_lo(gl[k][e]), bf16_hi(gl[k][e]), bf16_lo(ul[k][e]),
                           bf16_hi(ul[k][e]), a0, a1, b0, b1);
          wg[e] = f32_to_bf16_bits(a0) | (f32_to_bf16_bits(a1) << 16);
          wu[e] = f32_to_bf16_bits(b0) | (f32_to_bf16_bits(b1) << 16);
        }
        uint16_t *pg = static_cast<uint16_t *>(A.out) + (row0 + 4 * g + kb + k) * ld + c;
        st_cs_v8(pg, wg[0], wg[1], wg[2], wg[3], wg[4], wg[5], wg[6], wg[7]);
        st_cs_v8(pg + I, wu[0], wu[1], wu[2], wu[3], wu[4], wu[5], wu[6], wu[7]);
      }
    }
  }
}

// Bound of the waits that let a CTA leave cleanly: the producer's wait for its
// own copies to land and the MMA thread's wait for its own MMAs to finish.
// They are separate from the pipeline waits' limit (GemmArgs::wait_limit,
// which a test may shrink so that pipeline waits run out): the copies and
// MMAs in flight complete by themselves, and no CTA may leave (or free its
// tensor memory) before they have.
constexpr uint64_t kDrainLimit = (uint64_t)1 << 26;

// A bounded mbarrier wait that also gives up when another role of the CTA
// has raised the abort flag.  A wait that runs out raises the flag and records
// NV_ERR_TIMEOUT.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, uint64_t limit, volatile int *abort,
                                              int *status) {
  for (uint64_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 255 && *abort) return false;
  }
  *abort = 1;
  record_error(status, NV_ERR_TIMEOUT);
  return false;
}

// One output tile of the schedule.
struct Tile {
  int e, nk, a_row, b_row, mrows, k_off;
  int64_t a_tile, b_tile, k_atom0, out_row0, out_col0;
  int64_t sfb_g, sfb_u;  // SwiGLU kind: scale tiles of the gate and up rows
  int bh;                // SwiGLU kind: which 64-row half of those tiles
};

template <int KIND>
__device__ __forceinline__ Tile decode_tile(int t, const GemmArgs &A, const int *s_off, const int *s_pad) {
  Tile T;
  if (KIND == kGemmNvfp4FwdSwiglu) {
    // 128 rows x 64 hidden features: B = gate rows [64 nt, 64 nt + 64) over the
    // matching up rows (I further down the expert's w13)
    const int pm = t / A.ntn, nt = t - (t / A.ntn) * A.ntn;
    const int p0 = pm * 128;
    const int e = find_group(s_pad, A.E, p0);
    T.e = e;
    T.a_row = s_off[e] + (p0 - s_pad[e]);
    T.mrows = min(128, s_off[e + 1] - T.a_row);
    const int64_t g_row = (int64_t)e * 2 * A.I + (int64_t)nt * 64;
    T.b_row = (int)g_row;
    T.sfb_g = g_row / 128;
    T.sfb_u = (g_row + A.I) / 128;
    T.bh = nt & 1;  // I % 128 == 0: gate and up rows sit in the same half of their tiles
    T.a_tile = pm;
    T.b_tile = 0;
    T.nk = (int)(A.K / 256);
    T.k_off = 0;
    T.k_atom0 = 0;
    T.out_row0 = T.a_row;
    T.out_col0 = (int64_t)nt * 64;
  } else if (KIND != kGemmMxfp8Dw) {
    const int pm = t / A.ntn, nt = t - (t / A.ntn) * A.ntn;
    const int p0 = pm * 128;
    const int e = find_group(s_pad, A.E, p0);
    T.e = e;
    T.a_row = s_off[e] + (p0 - s_pad[e]);
    T.mrows = min(128, s_off[e + 1] - T.a_row);
    T.b_row = e * (int)(KIND == kGemmNvfp4Fwd ? A.N : A.K) + nt * kBN;
    T.a_tile = pm;
    T.b_tile = T.b_row / 128;
    T.nk = (int)(KIND == kGemmNvfp4Fwd ? A.K / 256 : A.N / 128);
    T.k_off = 0;
    T.k_atom0 = 0;
    T.out_row0 = T.a_row;
    T.out_col0 = (int64_t)nt * kBN;
  } else {
    const int per_e = A.ntm * A.ntn;
    const int e = t / per_e;
    const int r = t - e * per_e, mt = r / A.ntn, nt = r - (r / A.ntn) * A.ntn;
    T.e = e;
    T.a_row = mt * 128;
    T.b_row = nt * kBN;
    T.mrows = 128;
    T.nk = (s_pad[e + 1] - s_pad[e]) / 128;
    T.k_off = s_pad[e];
    T.a_tile = mt;
    T.b_tile = T.b_row / 128;
    T.k_atom0 = s_pad[e] / 128;
    T.out_row0 = (int64_t)e * A.N + (int64_t)mt * 128;
    T.out_col0 = (int64_t)nt * kBN;
  }
  return T;
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int KIND, int STAGES, int NACC, bool kS2f6 = false, bool kSwb = false>
__global__ void __launch_bounds__(192, 2)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmArgs A) {
  static_assert(!kSwb || KIND == kGemmMxfp8Dx, "the SwiGLU backward epilogue is the dgrad's");
  using C = Cfg<KIND, STAGES, NACC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t *sA = smem;
  uint8_t *sB = sA + STAGES * C::A_BYTES;
  uint8_t *sSFA = sB + STAGES * C::B_BYTES;
  uint8_t *sSFB = sSFA + STAGES * C::SFA_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sSFB + STAGES * C::SFB_BYTES);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + C::NBARS);
  volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
  int *s_flag = reinterpret_cast<int *>(s_tmem + 2);
  int *s_off = s_flag + 2;
  int *s_pad = s_off + (A.E + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!load_groups(A.groups, A.E, A.M_total, s_off, s_pad, s_flag, A.status)) return;
  const int num_tiles =
      KIND == kGemmMxfp8Dw ? A.E * A.ntm * A.ntn : (s_pad[A.E] / 128) * A.ntn;
  if ((int)blockIdx.x >= num_tiles) return;  // uniform over the CTA

  uint64_t *full = bars, *empty = bars + STAGES, *acc_full = bars + 2 * STAGES, *acc_empty = acc_full + NACC;
  uint64_t *mma_done = acc_empty + NACC;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(mma_done), 1);
    for (int s = 0; s < STAGES; ++s) {
      // SwiGLU kind: the 32 producer lanes' arrivals (their scale copies
      // landed and made visible to the tensor core) come on top of the TMA
      // transaction arrival
      mbar_init(smem_u32(&full[s]), KIND == kGemmNvfp4FwdSwiglu ? 33 : 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), 4);  // one arrival per epilogue warp
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(s_tmem), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 0 && (lane == 0 || KIND == kGemmNvfp4FwdSwiglu)) {
    // ---- producer (lane 0; the whole warp for the SwiGLU kind) ------------------
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
    }
    uint32_t it = 0;  // global stage counter of this CTA
    bool ok = true;
    for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
      const Tile T = decode_tile<KIND>(t, A, s_off, s_pad);
      for (int ks = 0; ks < T.nk; ++ks, ++it) {
        const uint32_t s = it % STAGES;
        if (it >= STAGES &&
            !wait_or_abort(smem_u32(&empty[s]), ((it / STAGES) - 1) & 1, A.wait_limit, s_abort, A.status)) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&full[s]);
        const int64_t katom = T.k_atom0 + (int64_t)ks * C::kAtomsPerStage;
        if (KIND == kGemmNvfp4FwdSwiglu) {
          if (lane == 0) {
            mbar_arrive_expect_tx(fb, C::STAGE_BYTES - C::SFB_BYTES);
            tma_load_2d(smem_u32(sA + s * C::A_BYTES), &tmA, T.k_off + ks * 128, T.a_row, fb);
            tma_load_2d(smem_u32(sB + s * C::B_BYTES), &tmB, T.k_off + ks * 128, T.b_row, fb);
            tma_load_2d(smem_u32(sB + s * C::B_BYTES + 64 * 128), &tmB, T.k_off + ks * 128, T.b_row + (int)A.I,
                        fb);
            bulk_load(smem_u32(sSFA + s * C::SFA_BYTES), A.a_scales + (T.a_tile * A.ka + katom) * 512,
                      C::SFA_BYTES, fb);
          }
          // the B scale tiles of the 64 gate + 64 up rows: row `lane` of each
          // 128x4 tile holds B rows lane, lane+32 (gate: 8 bytes of the gate
          // rows' tile) and lane+64, lane+96 (up: 8 bytes of the up rows' tile)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t dst = smem_u32(sSFB + s * C::SFB_BYTES + j * 512 + lane * 16);
            cp_async8(dst, A.b_scales + (T.sfb_g * A.ka + katom + j) * 512 + lane * 16 + 8 * T.bh);
            cp_async8(dst + 8, A.b_scales + (T.sfb_u * A.ka + katom + j) * 512 + lane * 16 + 8 * T.bh);
          }
          cp_async_commit();
          // one stage behind: the previous stage's copies have landed; the
          // proxy fence makes them visible to tcgen05.cp, then this lane
          // arrives on that stage's barrier (off the MMA thread's path)
          if (it >= 1) {
            cp_async_wait_prev_group();
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&full[(it - 1) % STAGES]));
          }
        } else {
          mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
          tma_load_2d(smem_u32(sA + s * C::A_BYTES), &tmA, T.k_off + ks * 128, T.a_row, fb);
          tma_load_2d(smem_u32(sB + s * C::B_BYTES), &tmB, T.k_off + ks * 128, T.b_row, fb);
          bulk_load(smem_u32(sSFA + s * C::SFA_BYTES), A.a_scales + (T.a_tile * A.ka + katom) * 512, C::SFA_BYTES,
                    fb);
#pragma unroll
          for (int j = 0; j < kBN / 128; ++j)
            bulk_load(smem_u32(sSFB + s * C::SFB_BYTES + j * C::SFA_BYTES),
                      A.b_scales + ((T.b_tile + j) * A.ka + katom) * 512, C::SFA_BYTES, fb);
        }
      }
    }
    if (KIND == kGemmNvfp4FwdSwiglu && it >= 1) {  // the last stage's scale copies
      cp_async_wait_all_groups();
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&full[(it - 1) % STAGES]));
    }
    // drain: every copy this thread issued has landed before the CTA leaves
    const uint32_t first = it > STAGES ? it - STAGES : 0;
    for (uint32_t k = first; k < it; ++k)
      if (!mbar_wait(smem_u32(&full[k % STAGES]), (k / STAGES) & 1, kDrainLimit)) {
        record_error(A.status, NV_ERR_TIMEOUT);
        break;
      }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ------------------------------------------------------------
    uint32_t it = 0, tc = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x, ++tc) {
      const Tile T = decode_tile<KIND>(t, A, s_off, s_pad);
      const uint32_t acc = tc % NACC, use = tc / NACC;
      // the accumulator's previous tile has been drained by the epilogue
      if (use >= 1 &&
          !wait_or_abort(smem_u32(&acc_empty[acc]), (use - 1) & 1, A.wait_limit, s_abort, A.status))
        break;
      tc_fence_after();
      const uint32_t d = tmem + acc * kBN;
      for (int ks = 0; ks < T.nk; ++ks, ++it) {
        const uint32_t s = it % STAGES;
        if (!wait_or_abort(smem_u32(&full[s]), (it / STAGES) & 1, A.wait_limit, s_abort, A.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sfa = tmem + C::ACC_COLS + s * C::SF_COLS;
        const uint32_t sfb = sfa + C::SFA_COLS;
        const uint32_t a_sf_smem = smem_u32(sSFA + s * C::SFA_BYTES);
        const uint32_t b_sf_smem = smem_u32(sSFB + s * C::SFB_BYTES);
#pragma unroll
        for (int j = 0; j < C::kAtomsPerStage; ++j) {
          tc_cp_sf(sfa + 4 * j, desc_sf(a_sf_smem + j * 512));
#pragma unroll
          for (int r = 0; r < kBN / 128; ++r)
            tc_cp_sf(sfb + j * (kBN / 32) + 4 * r, desc_sf(b_sf_smem + r * C::SFA_BYTES + j * 512));
        }
        const uint64_t da = desc_sw128(smem_u32(sA + s * C::A_BYTES));
        const uint64_t db = desc_sw128(smem_u32(sB + s * C::B_BYTES));
        if (C::kFp4) {
          // one 128-byte swizzle row holds 256 values: K = 96 at bytes 0
          // (scale blocks 0-5) and 48 (blocks 6-11, from byte 2 of the second
          // scale atom), K = 64 at byte 96 (blocks 12-15); an MMA must not
          // cross the row (K = 96 at byte 96 would)
          mma_nvf4_b16(d, da, db, C::IDESC | kIdescK96, sfa, sfb, ks != 0);
          mma_nvf4_b16(d, da + 3, db + 3, C::IDESC | kIdescK96 | idesc_sf_id(2), sfa + 4, sfb + (kBN / 32), 1u);
          mma_nvf4(d, da + 6, db + 6, C::IDESC, sfa + 12, sfb + 3 * (kBN / 32), 1u);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t accum = (ks | j) != 0;
            const uint32_t idesc = C::IDESC | ((uint32_t)j << 4) | ((uint32_t)j << 29);
            mma_mxf8(d, da + 2 * j, db + 2 * j, idesc, sfa, sfb, accum);
          }
        }
        tc_commit(smem_u32(&empty[s]));
      }
      tc_commit(smem_u32(&acc_full[acc]));  // arrives once this tile's MMAs are done (at once if none)
    }
    // every MMA and scale copy this thread issued has finished (also after an
    // abort) before tensor memory can be freed
    tc_commit(smem_u32(mma_done));
    if (!mbar_wait(smem_u32(mma_done), 0, kDrainLimit)) record_error(A.status, NV_ERR_TIMEOUT);
  } else if (warp >= 2) {
    // ---- epilogue ----------------------------------------------------------------
    const int q = warp & 3;
    const int row = q * 32 + lane;
    uint32_t tc = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tc) {
      const Tile T = decode_tile<KIND>(t, A, s_off, s_pad);
      const uint32_t acc = tc % NACC;
      if (kSwb && row < T.mrows) prefetch_swiglu_rows<kBN>(A, T.out_row0 + row, T.out_col0);
      if (!wait_or_abort(smem_u32(&acc_full[acc]), (tc / NACC) & 1, A.wait_limit, s_abort, A.status)) break;
      tc_fence_after();
      const bool store = row < T.mrows;
      const int64_t orow = T.out_row0 + row;
      float alpha = 1.0f;
      if (KIND == kGemmNvfp4Fwd || KIND == kGemmNvfp4FwdSwiglu)  // the row's own outer scale when per token
        alpha = __fmul_rn(A.a_sg_rows ? (store ? A.a_sg[orow] : 0.0f) : A.a_sg[0], A.b_sg[T.e]);
      // read the whole accumulator row into registers, release the
      // accumulator to the MMA thread, then convert and store
      uint32_t r[kBN];
      if (T.nk > 0) {
        const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + acc * kBN;
#pragma unroll
        for (int c0 = 0; c0 < kBN; c0 += 32) tmem_ld32_nowait(tb + (uint32_t)c0, &r[c0]);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < kBN; ++i) r[i] = 0u;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acc_empty[acc]));
      if (KIND == kGemmNvfp4FwdSwiglu) {
        // columns 0-63: gate, 64-127: up of hidden features out_col0 .. +63
        swiglu_epilogue(A, r, alpha, store, orow, T.out_col0, lane);
      } else if (kSwb) {  // dgrad with the SwiGLU backward: the warp's 32 rows together
        swiglu_bwd_epilogue<kBN>(A, r, T.out_row0 + q * 32, T.out_col0, lane, T.mrows - q * 32);
      } else if (KIND == kGemmMxfp8Dw && A.out_fp32) {
        // wgrad: the warp's 32 fp32 dW rows (all exist; alpha is 1) as whole lines
        uint8_t *row0 = static_cast<uint8_t *>(A.out) + ((T.out_row0 + q * 32) * A.out_ld + T.out_col0) * 4;
#pragma unroll
        for (int S = 0; S < kBN / 32; ++S) {
          uint32_t w[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) w[k] = r[32 * S + k];
          store_segment_coalesced(row0 + 128 * S, A.out_ld * 4, w, lane, T.mrows - q * 32);
        }
      } else if (store) {
        if constexpr (KIND == kGemmNvfp4Fwd && kS2f6) {
          // the combine direction's quantizer on the bf16 output rows: each
          // 32-column block of the row is rounded to bf16 exactly as the plain
          // output, then rotated and quantized as rht32_s2f6_quantize would
          uint16_t *dst = A.out ? static_cast<uint16_t *>(A.out) + orow * A.out_ld + T.out_col0 : nullptr;
#pragma unroll
          for (int blk = 0; blk < kBN / 32; ++blk) {
            uint32_t w[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
              w[k] = pack_bf16x2(__fmul_rn(__uint_as_float(r[32 * blk + 2 * k]), alpha),
                                 __fmul_rn(__uint_as_float(r[32 * blk + 2 * k + 1]), alpha));
            if (dst) {
              st_cs_v8(dst + 32 * blk, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
              st_cs_v8(dst + 32 * blk + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
            }
            uint32_t pk[8];
            const uint32_t sc = rht32_s2f6_block(w, A.rht, pk);
            st_cs_v8(A.s2f6_codes + orow * A.out_ld + T.out_col0 + 32 * blk, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5],
                     pk[6], pk[7]);
            A.s2f6_scales[orow * (A.out_ld / 32) + T.out_col0 / 32 + blk] = (uint8_t)sc;
          }
        } else if (A.out_fp32) {
          float *dst = static_cast<float *>(A.out) + orow * A.out_ld + T.out_col0;
#pragma unroll
          for (int i = 0; i < kBN; i += 8) {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(__fmul_rn(__uint_as_float(r[i + k]), alpha));
            st_cs_v8(dst + i, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
          }
        } else {
          uint16_t *dst = static_cast<uint16_t *>(A.out) + orow * A.out_ld + T.out_col0;
#pragma unroll
          for (int i = 0; i < kBN; i += 16) {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              w[k] = pack_bf16x2(__fmul_rn(__uint_as_float(r[i + 2 * k]), alpha),
                                 __fmul_rn(__uint_as_float(r[i + 2 * k + 1]), alpha));
            st_cs_v8(dst + i, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
          }
        }
      }
    }
  }
  __syncwarp();  // single-lane roles rejoin their warps before the CTA barrier
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// CTA-pair variant (cta_group::2): one 256 x 256 output tile per pair of SMs.
// Each CTA of the pair stages 128 rows of A and its 128-row half of B; one
// thread of the even CTA issues M=256, N=256 MMAs that read both CTAs' shared
// memory and accumulate 128 rows x 256 columns in each CTA's tensor memory.
// Per FLOP this moves half the L2 -> SM operand bytes of the 128 x 128 tile.
// The odd CTA's TMA loads signal the even CTA's "full" barrier; the MMA
// commits arrive on both CTAs' barriers (multicast); the odd CTA's epilogue
// warps release the accumulator on the even CTA's barrier.  The block-scale
// tiles are loaded with TMA too (2-D view of the scale buffer, 128-byte rows)
// so that they can signal the peer's barrier; each CTA holds the scales of
// its own A rows and of all 256 B rows.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4}], [%5];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_5d_pair(uint32_t dst, const CUtensorMap *map, int x, int y, int z, int w,
                                                 int v, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4, %5, %6}], [%7];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(v), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap *map, int x, int y, int z, int w,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4, %5}], [%6];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}
// completion of this thread's earlier pair MMAs, signalled on this CTA's barrier only
__device__ __forceinline__ void tc_commit_pair_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_cp_sf_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void mma_nvf4_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                              uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ void mma_nvf4_pair_b16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                                  uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.block16 [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ void mma_mxf8_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                              uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
// Relaxed: the only ordering needed is that this warp's tensor-memory loads
// have completed (tcgen05.wait::ld), not that its earlier global stores are
// visible, so no release fence is paid here.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Output tile of a CTA pair: 256 x BN.  BN = 256: one pair per SM pair (the
// 256-column accumulator fills half of each SM's tensor memory); BN = 128: two
// pairs per SM pair, so one pair's epilogue runs under the other's MMAs, with
// half the scale copies per FLOP of the 128 x 128 kernel.
//
// A ring stage holds CHUNKS k-chunks of 128 bytes per operand row.  Every
// barrier wait of the MMA issuer leaves the tensor pipe idle for about 200
// cycles (measured: the pipe queues almost nothing ahead of the issuing
// thread), so the MXFP8 kernels take two chunks (8 MMAs) per wait in three
// stages rather than one chunk per wait in six: the same shared memory and
// bytes in flight, half the waits.  A tile's last stage may hold one chunk.
template <int KIND, int STAGES, int BN, int CHUNKS = 1>
struct CfgPair {
  static_assert(BN == 128 || BN == 256, "pair tile width");
  static_assert(KIND != kGemmNvfp4FwdSwiglu || BN == 256, "SwiGLU pair tiles: 128 gate + 128 up rows");
  static constexpr bool kFp4 = KIND == kGemmNvfp4Fwd || KIND == kGemmNvfp4FwdSwiglu;
  static constexpr int kAtomsPerStage = kFp4 ? 4 : 1;   // 128x4 scale tiles per 128 rows per chunk
  static constexpr int kBHalf = BN / 2;                 // B rows staged by each CTA
  static constexpr int kSfbTiles = BN / 128;            // 128-row scale tiles of B per k-atom
  static constexpr int A_CHUNK = 128 * 128;
  static constexpr int B_CHUNK = kBHalf * 128;          // this CTA's half of B
  static constexpr int SFA_CHUNK = kAtomsPerStage * 512;
  static constexpr int SFB_CHUNK = kSfbTiles * SFA_CHUNK;  // scales of all BN rows of B
  static constexpr int CHUNK_BYTES = A_CHUNK + B_CHUNK + SFA_CHUNK + SFB_CHUNK;
  static constexpr int A_BYTES = CHUNKS * A_CHUNK;
  static constexpr int B_BYTES = CHUNKS * B_CHUNK;
  static constexpr int SFA_BYTES = CHUNKS * SFA_CHUNK;
  static constexpr int SFB_BYTES = CHUNKS * SFB_CHUNK;
  static constexpr int STAGE_BYTES = CHUNKS * CHUNK_BYTES;
  static constexpr int SFA_COLS = kAtomsPerStage * 4;   // per chunk
  static constexpr int SFB_COLS = kAtomsPerStage * (BN / 32);
  static constexpr int SF_CHUNK_COLS = SFA_COLS + SFB_COLS;
  static constexpr int SF_COLS = CHUNKS * SF_CHUNK_COLS;  // per stage
  static constexpr int ACC_COLS = BN;
  static constexpr int TMEM_COLS = cpow2(ACC_COLS + STAGES * SF_COLS);
  // full, empty, acc_full, acc_empty, mma_done, then (with copy issuers)
  // sf_land per stage and one drain barrier per issuer
  static constexpr int kCtasPerSm = BN == 128 ? 2 : 1;
  // A tcgen05.cp holds its issuing thread for about 64 cycles and runs
  // alongside the MMAs only when another thread issues it, so with one pair
  // per SM pair (room for two more warps) two warps of the even CTA issue a
  // stage's scale copies, half each, while the MMA thread issues its MMAs.
  // The 256 x 128 variant (two pairs per SM pair) keeps the copies on the MMA
  // thread: its registers leave no room for more warps.
  static constexpr int kSfWarps = kCtasPerSm == 1 ? 2 : 0;
  static constexpr int NBARS = 2 * STAGES + 3 + (kSfWarps ? STAGES + kSfWarps : 0);
  static constexpr int kEpi0 = 2 + kSfWarps;            // first epilogue warp
  // Wide loads (two-chunk stages with copy issuers): a stage's two k-chunks
  // come in one load per tensor (A, B: 3-D boxes of two 128-byte k-chunks;
  // A scales: the two chunks' rows; B scales: a 5-D box [chunk][tile][rows]),
  // four loads a stage instead of eight -- a thread issuing TMA loads gets
  // about 46 B/clk whatever the box size.  A stage holding one chunk (the
  // last of an odd count) still loads two; the second is not used.
  static constexpr bool kWideLoads = CHUNKS == 2 && kSfWarps > 0;
  static constexpr int kEpiWarps = BN / 32;             // per lane quadrant: BN / 128 warps of 128 columns
  static constexpr int kThreads = 32 * (kEpi0 + kEpiWarps);
  static constexpr uint32_t IDESC = (kFp4 ? ((1u << 7) | (1u << 10)) : (1u << 23)) |
                                    ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
  static size_t smem_bytes(int E) {
    return 1024 + (size_t)STAGES * STAGE_BYTES + NBARS * 8 + 32 + (size_t)(E + 1) * 16 + 64;
  }
  static_assert(TMEM_COLS * kCtasPerSm <= 512, "tensor memory");
};

// Wgrad tile order.  D lists the tiles expert by expert in decreasing padded
// token count (a tile's MMA time grows with its expert's tokens; every tile
// stores the same 256 x 256 fp32 block).  Pair p takes D[r * P + p] in round
// r, with every odd round walked in reverse (position r * P + P - 1 - p), so
// that the pairs' sums of tile times stay within about 1% of each other (the
// last, partial round is not reversed).  At most two experts' operands are
// live at a time; within an expert the tiles go column-major when A has fewer
// row blocks than B, else row-major (decode_pair).
__device__ __forceinline__ int dw_sorted_index(int t, int pair, int npairs, int T) {
  const int r = t / npairs;
  if ((r & 1) && (r + 1) * npairs <= T) return r * npairs + (npairs - 1 - pair);
  return t;
}

// s_ord[k]: the expert with the k-th largest padded token count (ties: lower
// index first).  Every thread of the CTA must call it.
__device__ inline void sort_experts_by_size(const int *s_pad, int E, int *s_ord) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int pe = s_pad[e + 1] - s_pad[e];
    int rank = 0;
    for (int f = 0; f < E; ++f) {
      const int pf = s_pad[f + 1] - s_pad[f];
      rank += (pf > pe) || (pf == pe && f < e);
    }
    s_ord[rank] = e;
  }
  __syncthreads();
}

// One pair tile, seen from CTA `cta` (0 or 1) of the pair.
struct PairTile {
  int e, nk, k_off, mrows;
  int a_row, b_row;
  int64_t a_tile, k_atom0, out_row0, out_col0;
  int64_t b_sft[2];  // 128-row scale tiles of the tile's B rows
};

// s_pb[e]: number of 256-row pair blocks before expert e (fwd, dgrad);
// s_ord: experts by decreasing size (wgrad)
template <int KIND, int BN>
__device__ __forceinline__ PairTile decode_pair(int t, const GemmArgs &A, const int *s_off, const int *s_pad,
                                                const int *s_pb, const int *s_ord, int pair, int npairs,
                                                int num_tiles, int cta) {
  PairTile T;
  if (KIND != kGemmMxfp8Dw) {
    const int pm = t / A.ntn, nt = t - (t / A.ntn) * A.ntn;
    const int e = find_group(s_pb, A.E, pm);
    const int p0 = s_pad[e] + (pm - s_pb[e]) * 256;
    int ph = p0 + 128 * cta;
    const bool live = ph < s_pad[e + 1];
    if (!live) ph = p0;  // an empty half re-reads the first half; nothing of it is stored
    T.e = e;
    T.a_row = s_off[e] + (ph - s_pad[e]);
    T.mrows = live ? min(128, s_off[e + 1] - T.a_row) : 0;
    T.a_tile = ph / 128;
    constexpr bool kFwd = KIND == kGemmNvfp4Fwd || KIND == kGemmNvfp4FwdSwiglu;
    const int nb = (int)(kFwd ? A.N : A.K);
    if (KIND == kGemmNvfp4FwdSwiglu) {
      // 128 hidden features: the even CTA stages their 128 gate rows, the odd
      // CTA the matching up rows (I further down the expert's w13), so that
      // accumulator columns 0-127 are the gate and 128-255 the up
      const int64_t g_row = (int64_t)e * nb + (int64_t)nt * 128;
      T.b_row = (int)(g_row + (int64_t)cta * A.I);
      T.b_sft[0] = g_row / 128;
      T.b_sft[1] = (g_row + A.I) / 128;
      T.out_col0 = (int64_t)nt * 128;
    } else {
      T.b_row = e * nb + nt * BN + (BN / 2) * cta;
      T.b_sft[0] = ((int64_t)e * nb + (int64_t)nt * BN) / 128;
      T.b_sft[1] = T.b_sft[0] + 1;
      T.out_col0 = (int64_t)nt * BN;
    }
    T.nk = (int)(kFwd ? A.K / 256 : A.N / 128);
    T.k_off = 0;
    T.k_atom0 = 0;
    T.out_row0 = T.a_row;
  } else {
    const int per_e = A.ntm * A.ntn;
    const int d = dw_sorted_index(t, pair, npairs, num_tiles);
    const int k = d / per_e;
    const int e = s_ord[k];
    // within the expert, the operand with fewer 256-row blocks is swept in
    // the inner loop: the ~38 tiles of an expert in flight at a time then
    // read all of its blocks (which stay in the L2 from one round to the
    // next) and only a few blocks of the other operand, each once
    const int r = d - k * per_e;
    int mt, nt;
    if (A.ntm < A.ntn) {  // column-major
      nt = r / A.ntm;
      mt = r - nt * A.ntm;
    } else {  // row-major
      mt = r / A.ntn;
      nt = r - mt * A.ntn;
    }
    T.e = e;
    T.a_row = mt * 256 + 128 * cta;
    T.b_row = nt * BN + (BN / 2) * cta;
    T.mrows = 128;
    T.nk = (s_pad[e + 1] - s_pad[e]) / 128;
    T.k_off = s_pad[e];
    T.a_tile = T.a_row / 128;
    T.b_sft[0] = (int64_t)nt * (BN / 128);
    T.b_sft[1] = T.b_sft[0] + 1;
    T.k_atom0 = s_pad[e] / 128;
    T.out_row0 = (int64_t)e * A.N + T.a_row;
    T.out_col0 = (int64_t)nt * BN;
  }
  return T;
}

// warp 0: exclusive scan of ceil(padded group size / 256) into s_pb[0..E]
__device__ inline void scan_pair_blocks(const int *s_pad, int E, int *s_pb) {
  if (threadIdx.x < 32) {
    int carry = 0;
    for (int base = 0; base <= E; base += 32) {
      const int e = base + (int)threadIdx.x;
      int v = 0;
      if (e < E) v = (s_pad[e + 1] - s_pad[e] + 255) / 256;
      int incl = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if ((int)threadIdx.x >= d) incl += n;
      }
      if (e <= E) s_pb[e] = carry + incl - v;
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
  __syncthreads();
}

// A bounded wait that raises the abort flag of both CTAs of the pair when it
// runs out (or gives up when one of them is raised).
__device__ __forceinline__ bool wait_pair(uint32_t bar, uint32_t parity, uint64_t limit, volatile int *abort,
                                          uint32_t peer_abort, int *status) {
  for (uint64_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 255 && *abort) return false;
  }
  *abort = 1;
  st_cluster_u32(peer_abort, 1u);
  record_error(status, NV_ERR_TIMEOUT);
  return false;
}

// The scale copies of one ring stage into its tensor-memory buffer: the A
// tiles (4 columns each) then the B tiles of each k-atom, numbered in that
// order over the stage's chunks; `part` < 0 issues all of them, else issuer
// `part` issues those with (number % kSfWarps) == part.
template <class C, int BN, int CHUNKS>
__device__ __forceinline__ void issue_stage_sf_copies(uint32_t tmem, uint32_t s, int nc, uint32_t a_sf_stage,
                                                      uint32_t b_sf_stage, int part) {
  constexpr int kParts = C::kSfWarps > 0 ? C::kSfWarps : 1;
  int k = 0;
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) {
    if (c >= nc) break;
    const uint32_t sfa = tmem + C::ACC_COLS + s * C::SF_COLS + c * C::SF_CHUNK_COLS;
    const uint32_t sfb = sfa + C::SFA_COLS;
    const uint32_t a_sf_smem = a_sf_stage + c * C::SFA_CHUNK;
    const uint32_t b_sf_smem = b_sf_stage + c * C::SFB_CHUNK;
#pragma unroll
    for (int j = 0; j < C::kAtomsPerStage; ++j) {
      if (part < 0 || k % kParts == part) tc_cp_sf_pair(sfa + 4 * j, desc_sf(a_sf_smem + j * 512));
      ++k;
#pragma unroll
      for (int r = 0; r < C::kSfbTiles; ++r) {
        if (part < 0 || k % kParts == part)
          tc_cp_sf_pair(sfb + j * (BN / 32) + 4 * r, desc_sf(b_sf_smem + r * C::SFA_CHUNK + j * 512));
        ++k;
      }
    }
  }
}

template <int KIND, int STAGES, int BN, int CHUNKS, bool kSwb = false>
__global__ void __launch_bounds__(CfgPair<KIND, STAGES, BN, CHUNKS>::kThreads,
                                  CfgPair<KIND, STAGES, BN, CHUNKS>::kCtasPerSm)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                             GemmArgs A) {
  static_assert(!kSwb || KIND == kGemmMxfp8Dx, "the SwiGLU backward epilogue is the dgrad's");
  using C = CfgPair<KIND, STAGES, BN, CHUNKS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t *sA = smem;
  uint8_t *sB = sA + STAGES * C::A_BYTES;
  uint8_t *sSFA = sB + STAGES * C::B_BYTES;
  uint8_t *sSFB = sSFA + STAGES * C::SFA_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sSFB + STAGES * C::SFB_BYTES);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + C::NBARS);
  volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
  int *s_flag = reinterpret_cast<int *>(s_tmem + 2);
  int *s_off = s_flag + 2;
  int *s_pad = s_off + (A.E + 1);
  int *s_pb = s_pad + (A.E + 1);
  int *s_ord = s_pb + (A.E + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = (int)cluster_ctarank();
  const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
  // identical in both CTAs of the pair, so an early return is taken by both
  if (!load_groups(A.groups, A.E, A.M_total, s_off, s_pad, s_flag, A.status)) return;
  scan_pair_blocks(s_pad, A.E, s_pb);
  if (KIND == kGemmMxfp8Dw) sort_experts_by_size(s_pad, A.E, s_ord);
  const int num_tiles = KIND == kGemmMxfp8Dw ? A.E * A.ntm * A.ntn : s_pb[A.E] * A.ntn;
  if (pair >= num_tiles) return;

  uint64_t *full = bars, *empty = bars + STAGES, *acc_full = bars + 2 * STAGES, *acc_empty = acc_full + 1;
  uint64_t *mma_done = acc_empty + 1;
  // with copy issuers: sf_land (a stage's scale tiles have landed, loaded
  // ahead of its operand tiles) and sf_done; a stage's "full" barrier then
  // also takes one commit per issuer, completing once its operand tiles have
  // landed and its scale tiles are in tensor memory, so that the MMA thread
  // waits once per stage (each wait idles the tensor pipe ~200 cycles)
  uint64_t *sf_land = mma_done + 1, *sf_done = sf_land + STAGES;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(mma_done), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1 + C::kSfWarps);  // the producer's arrival (+ one commit per issuer)
      mbar_init(smem_u32(&empty[s]), 1);
      if (C::kSfWarps) mbar_init(smem_u32(&sf_land[s]), 1);
    }
    for (int w = 0; w < C::kSfWarps; ++w) mbar_init(smem_u32(&sf_done[w]), 1);
    mbar_init(smem_u32(acc_full), 1);
    mbar_init(smem_u32(acc_empty), 2 * C::kEpiWarps);  // every epilogue warp of both CTAs
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(s_tmem), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // barriers of both CTAs initialised before any remote use
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t peer_abort = mapa_shared(smem_u32((const void *)s_abort), (uint32_t)(cta ^ 1));

  if (warp == 0 && lane == 0) {
    // ---- producer (both CTAs) ----------------------------------------------------
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmSA) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmSB) : "memory");
    uint32_t it = 0;
    bool ok = true;
    for (int t = pair; ok && t < num_tiles; t += npairs) {
      const PairTile T = decode_pair<KIND, BN>(t, A, s_off, s_pad, s_pb, s_ord, pair, npairs, num_tiles, cta);
      for (int ks = 0; ks < T.nk; ks += CHUNKS, ++it) {
        const uint32_t s = it % STAGES;
        const int nc = T.nk - ks < CHUNKS ? T.nk - ks : CHUNKS;
        if (it >= STAGES &&
            !wait_pair(smem_u32(&empty[s]), ((it / STAGES) - 1) & 1, A.wait_limit, s_abort, peer_abort, A.status)) {
          ok = false;
          break;
        }
        if constexpr (C::kWideLoads) {
          const uint32_t f0 = smem_u32(&full[s]), l0 = smem_u32(&sf_land[s]);
          if (cta == 0) {
            mbar_arrive_expect_tx(l0, 2 * 2 * (C::SFA_CHUNK + C::SFB_CHUNK));
            mbar_arrive_expect_tx(f0, 2 * 2 * (C::A_CHUNK + C::B_CHUNK));
          }
          const uint32_t lb = cta == 0 ? l0 : mapa_shared(l0, 0), fb = cta == 0 ? f0 : mapa_shared(f0, 0);
          const int64_t katom = T.k_atom0 + (int64_t)ks * C::kAtomsPerStage;
          tma_load_2d_pair(smem_u32(sSFA + s * C::SFA_BYTES), &tmSA, 0, (int)((T.a_tile * A.ka + katom) * 4), lb);
          tma_load_5d_pair(smem_u32(sSFB + s * C::SFB_BYTES), &tmSB, 0, 0, 0, (int)katom, (int)T.b_sft[0], lb);
          tma_load_3d_pair(smem_u32(sA + s * C::A_BYTES), &tmA, 0, T.a_row, T.k_off / 128 + ks, fb);
          tma_load_3d_pair(smem_u32(sB + s * C::B_BYTES), &tmB, 0, T.b_row, T.k_off / 128 + ks, fb);
          continue;
        }
        const uint32_t fb_local = smem_u32(&full[s]);
        const uint32_t fb = cta == 0 ? fb_local : mapa_shared(fb_local, 0);
        // with copy issuers the scale tiles go first, on their own barrier,
        // so that their copies to tensor memory overlap the operand loads
        const uint32_t sb_local = C::kSfWarps ? smem_u32(&sf_land[s]) : fb_local;
        const uint32_t sb = cta == 0 ? sb_local : mapa_shared(sb_local, 0);
        constexpr int kSfBytes = C::SFA_CHUNK + C::SFB_CHUNK;
        if (cta == 0) {
          if (C::kSfWarps) {
            mbar_arrive_expect_tx(sb_local, 2 * nc * kSfBytes);
            mbar_arrive_expect_tx(fb_local, 2 * nc * (C::CHUNK_BYTES - kSfBytes));
          } else {
            mbar_arrive_expect_tx(fb_local, 2 * nc * C::CHUNK_BYTES);
          }
        }
        for (int c = 0; c < nc; ++c) {
          const int64_t katom = T.k_atom0 + (int64_t)(ks + c) * C::kAtomsPerStage;
          tma_load_2d_pair(smem_u32(sSFA + s * C::SFA_BYTES + c * C::SFA_CHUNK), &tmSA, 0,
                           (int)((T.a_tile * A.ka + katom) * 4), sb);
          if (C::kSfbTiles == 2) {  // both scale tiles of the B rows in one load (tmSB: 4-D view)
            tma_load_4d_pair(smem_u32(sSFB + s * C::SFB_BYTES + c * C::SFB_CHUNK), &tmSB, 0, (int)(katom * 4), 0,
                             (int)T.b_sft[0], sb);
          } else {
            tma_load_2d_pair(smem_u32(sSFB + s * C::SFB_BYTES + c * C::SFB_CHUNK), &tmSB, 0,
                             (int)((T.b_sft[0] * A.ka + katom) * 4), sb);
          }
        }
        for (int c = 0; c < nc; ++c) {
          const int k = ks + c;
          tma_load_2d_pair(smem_u32(sA + s * C::A_BYTES + c * C::A_CHUNK), &tmA, T.k_off + k * 128, T.a_row, fb);
          tma_load_2d_pair(smem_u32(sB + s * C::B_BYTES + c * C::B_CHUNK), &tmB, T.k_off + k * 128, T.b_row, fb);
        }
      }
    }
    if (cta == 0) {  // the even CTA's barriers count both CTAs' bytes: wait for the last copies
      const uint32_t first = it > STAGES ? it - STAGES : 0;
      for (uint32_t k = first; k < it; ++k)
        if (!mbar_wait(smem_u32(&full[k % STAGES]), (k / STAGES) & 1, kDrainLimit) ||
            (C::kSfWarps && !mbar_wait(smem_u32(&sf_land[k % STAGES]), (k / STAGES) & 1, kDrainLimit))) {
          record_error(A.status, NV_ERR_TIMEOUT);
          break;
        }
    }
  } else if (warp == 1 && lane == 0 && cta == 0) {
    // ---- MMA issuer (even CTA only) ---------------------------------------------
    uint32_t it = 0, tc = 0;
    bool ok = true;
    for (int t = pair; ok && t < num_tiles; t += npairs, ++tc) {
      const PairTile T = decode_pair<KIND, BN>(t, A, s_off, s_pad, s_pb, s_ord, pair, npairs, num_tiles, 0);
      if (tc >= 1 && !wait_pair(smem_u32(acc_empty), (tc - 1) & 1, A.wait_limit, s_abort, peer_abort, A.status))
        break;
      tc_fence_after();
      for (int ks = 0; ks < T.nk; ks += CHUNKS, ++it) {
        const uint32_t s = it % STAGES;
        const int nc = T.nk - ks < CHUNKS ? T.nk - ks : CHUNKS;
        if (!wait_pair(smem_u32(&full[s]), (it / STAGES) & 1, A.wait_limit, s_abort, peer_abort, A.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (!C::kSfWarps)
          issue_stage_sf_copies<C, BN, CHUNKS>(tmem, s, nc, smem_u32(sSFA + s * C::SFA_BYTES),
                                               smem_u32(sSFB + s * C::SFB_BYTES), -1);
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c) {
          if (c >= nc) break;
          const uint32_t sfa = tmem + C::ACC_COLS + s * C::SF_COLS + c * C::SF_CHUNK_COLS;
          const uint32_t sfb = sfa + C::SFA_COLS;
          const uint64_t da = desc_sw128(smem_u32(sA + s * C::A_BYTES + c * C::A_CHUNK));
          const uint64_t db = desc_sw128(smem_u32(sB + s * C::B_BYTES + c * C::B_CHUNK));
          if (C::kFp4) {  // K = 96, 96, 64 per 128-byte row, as in the one-CTA kernel
            mma_nvf4_pair_b16(tmem, da, db, C::IDESC | kIdescK96, sfa, sfb, (ks + c) != 0);
            mma_nvf4_pair_b16(tmem, da + 3, db + 3, C::IDESC | kIdescK96 | idesc_sf_id(2), sfa + 4, sfb + (BN / 32),
                              1u);
            mma_nvf4_pair(tmem, da + 6, db + 6, C::IDESC, sfa + 12, sfb + 3 * (BN / 32), 1u);
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t accum = ((ks + c) | j) != 0;
              const uint32_t idesc = C::IDESC | ((uint32_t)j << 4) | ((uint32_t)j << 29);
              mma_mxf8_pair(tmem, da + 2 * j, db + 2 * j, idesc, sfa, sfb, accum);
            }
          }
        }
        tc_commit_pair(smem_u32(&empty[s]));
      }
      tc_commit_pair(smem_u32(acc_full));  // both CTAs: this tile's accumulator is complete
    }
    // every MMA and scale copy this thread issued (for both CTAs) has finished,
    // also after an abort, before either CTA frees its tensor memory (both
    // pass the cluster barrier below first)
    tc_commit_pair_local(smem_u32(mma_done));
    if (!mbar_wait(smem_u32(mma_done), 0, kDrainLimit)) record_error(A.status, NV_ERR_TIMEOUT);
  } else if (warp >= 2 && warp < C::kEpi0) {
    // ---- scale-copy issuers (even CTA only) ------------------------------------------
    // each stage, once its scale tiles have landed: this issuer's half of
    // the stage's copies, then a commit on the stage's full barrier, which
    // completes when both halves have been written to tensor memory (and the
    // stage's operand tiles have landed).  A
    // stage's buffer is rewritten only after its refill has landed, i.e.
    // after the MMAs that read it have completed (the producer refills a
    // stage after its MMAs' commit).
    if (lane == 0 && cta == 0) {
      const int part = warp - 2;
      uint32_t it = 0;
      bool ok = true;
      for (int t = pair; ok && t < num_tiles; t += npairs) {
        const PairTile T = decode_pair<KIND, BN>(t, A, s_off, s_pad, s_pb, s_ord, pair, npairs, num_tiles, 0);
        for (int ks = 0; ks < T.nk; ks += CHUNKS, ++it) {
          const uint32_t s = it % STAGES;
          const int nc = T.nk - ks < CHUNKS ? T.nk - ks : CHUNKS;
          if (!wait_pair(smem_u32(&sf_land[s]), (it / STAGES) & 1, A.wait_limit, s_abort, peer_abort, A.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_stage_sf_copies<C, BN, CHUNKS>(tmem, s, nc, smem_u32(sSFA + s * C::SFA_BYTES),
                                               smem_u32(sSFB + s * C::SFB_BYTES), part);
          tc_commit_pair_local(smem_u32(&full[s]));
        }
      }
      // every copy this thread issued has landed before tensor memory is freed
      tc_commit_pair_local(smem_u32(&sf_done[part]));
      if (!mbar_wait(smem_u32(&sf_done[part]), 0, kDrainLimit)) record_error(A.status, NV_ERR_TIMEOUT);
    }
  } else if (warp >= C::kEpi0) {
    // ---- epilogue (both CTAs): BN / 32 warps, 128 columns each ------------------------
    const int q = warp & 3;
    const int half = (warp - C::kEpi0) >> 2;
    const int row = q * 32 + lane;
    const uint32_t acc_empty_addr = cta == 0 ? smem_u32(acc_empty) : mapa_shared(smem_u32(acc_empty), 0);
    uint32_t tc = 0;
    for (int t = pair; t < num_tiles; t += npairs, ++tc) {
      const PairTile T = decode_pair<KIND, BN>(t, A, s_off, s_pad, s_pb, s_ord, pair, npairs, num_tiles, cta);
      if (kSwb && row < T.mrows) prefetch_swiglu_rows<128>(A, T.out_row0 + row, T.out_col0 + half * 128);
      if (!wait_pair(smem_u32(acc_full), tc & 1, A.wait_limit, s_abort, peer_abort, A.status)) break;
      tc_fence_after();
      const bool store = row < T.mrows;
      const int64_t orow = T.out_row0 + row;
      float alpha = 1.0f;
      if (C::kFp4) alpha = __fmul_rn(A.a_sg_rows ? (store ? A.a_sg[orow] : 0.0f) : A.a_sg[0], A.b_sg[T.e]);
      const int64_t ocol = T.out_col0 + half * 128;
      uint32_t r[128];
      if (T.nk > 0) {
        const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16);
        if (KIND == kGemmNvfp4FwdSwiglu) {  // gate columns half*64 .. +63, then the matching up columns
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 32) {
            tmem_ld32_nowait(tb + (uint32_t)(half * 64 + c0), &r[c0]);
            tmem_ld32_nowait(tb + (uint32_t)(128 + half * 64 + c0), &r[64 + c0]);
          }
        } else {
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 32) tmem_ld32_nowait(tb + (uint32_t)(half * 128 + c0), &r[c0]);
        }
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 128; ++i) r[i] = 0u;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (cta == 0)
          mbar_arrive(acc_empty_addr);
        else
          mbar_arrive_cluster(acc_empty_addr);
      }
      if (KIND == kGemmNvfp4FwdSwiglu) {
        swiglu_epilogue(A, r, alpha, store, orow, T.out_col0 + half * 64, lane);
      } else if (kSwb) {  // dgrad with the SwiGLU backward: the warp's 32 rows together
        swiglu_bwd_epilogue<128>(A, r, T.out_row0 + q * 32, ocol, lane, T.mrows - q * 32);
      } else if (KIND == kGemmMxfp8Dw && A.out_fp32) {
        // wgrad: fp32 dW rows are 512 bytes per lane and the stores are the
        // epilogue's bottleneck, so the warp writes them as whole lines (the
        // tile's 128 rows all exist; alpha is 1)
        uint8_t *row0 = static_cast<uint8_t *>(A.out) + ((T.out_row0 + q * 32) * A.out_ld + ocol) * 4;
#pragma unroll
        for (int S = 0; S < 4; ++S) {
          uint32_t w[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) w[k] = r[32 * S + k];
          store_segment_coalesced(row0 + 128 * S, A.out_ld * 4, w, lane, T.mrows - q * 32);
        }
      } else if (store) {
        if (A.out_fp32) {
          float *dst = static_cast<float *>(A.out) + orow * A.out_ld + ocol;
#pragma unroll
          for (int i = 0; i < 128; i += 8) {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(__fmul_rn(__uint_as_float(r[i + k]), alpha));
            st_cs_v8(dst + i, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
          }
        } else {
          uint16_t *dst = static_cast<uint16_t *>(A.out) + orow * A.out_ld + ocol;
#pragma unroll
          for (int i = 0; i < 128; i += 16) {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              w[k] = pack_bf16x2(__fmul_rn(__uint_as_float(r[i + 2 * k]), alpha),
                                 __fmul_rn(__uint_as_float(r[i + 2 * k + 1]), alpha));
            st_cs_v8(dst + i, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
          }
        }
      }
    }
  }
  // single-lane roles rejoin their warps first: an aligned barrier reached
  // by part of a warp must not let the CTA (or its peer) move on
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its peer may still signal it or read its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D byte matrix [outer][inner] (row stride `ld` bytes), box 128 bytes x box_rows
static bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A scale buffer of `bytes` bytes (a multiple of 512) viewed as rows of 128
// bytes; one box is `box_rows` rows (4 rows = one 512-byte 128x4 tile).
static bool make_sf_map(CUtensorMap *m, const void *base, uint64_t bytes, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, bytes / 128};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The B scale buffer as [tile][pair member z][ka * 4 rows of 128 bytes]:
// element (x, y, z, w) is byte x of row y of scale tile w + z * gap, so one
// box {128, rows, 2, 1} loads the same rows of two tiles `gap` tiles apart
// (consecutive tiles, or the gate and up tiles of the SwiGLU kind).
static bool make_sf_map_pair(CUtensorMap *m, const void *base, uint64_t n_tiles, uint64_t ka, uint64_t gap,
                             uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn || n_tiles <= gap) return false;
  const uint64_t tile_bytes = ka * 512;
  cuuint64_t dims[4] = {128, ka * 4, 2, n_tiles - gap};
  cuuint64_t strides[3] = {128, gap * tile_bytes, tile_bytes};
  cuuint32_t box[4] = {128, box_rows, 2, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Wide-load views: codes as [k-chunk][row][128 bytes] (box of two k-chunks,
// 128-byte swizzle), and B scales as [tile][k-chunk][pair member][rows of
// one chunk][128 bytes] (box: both members' rows of two k-chunks).
static bool make_map_chunks(CUtensorMap *m, const void *base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, rows, row_bytes / 128};
  cuuint64_t strides[2] = {row_bytes, 128};
  cuuint32_t box[3] = {128, box_rows, 2};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
static bool make_sf_map_pair_chunks(CUtensorMap *m, const void *base, uint64_t n_tiles, uint64_t ka, uint64_t gap,
                                    uint32_t chunk_rows) {
  auto fn = encode_fn();
  const uint64_t rows = ka * 4;  // 128-byte rows of one tile's scale block
  if (!fn || n_tiles <= gap || rows % chunk_rows) return false;
  const uint64_t tile_bytes = ka * 512;
  cuuint64_t dims[5] = {128, chunk_rows, 2, rows / chunk_rows, n_tiles - gap};
  cuuint64_t strides[4] = {128, gap * tile_bytes, (uint64_t)chunk_rows * 128, tile_bytes};
  cuuint32_t box[5] = {128, chunk_rows, 2, 2, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int num_sms() {
  static int n[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!n[dev] && cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n[dev] = 0;
  return n[dev];
}

template <int KIND, int STAGES, int NACC, bool kS2f6 = false, bool kSwb = false>
static int run(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &args, int64_t max_tiles,
               cudaStream_t s) {
  using C = Cfg<KIND, STAGES, NACC>;
  const size_t sm = C::smem_bytes(args.E);
  auto k = grouped_gemm_kernel<KIND, STAGES, NACC, kS2f6, kSwb>;
  static size_t attr_bytes = 0;  // largest dynamic shared memory requested so far
  if (sm > attr_bytes) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess)
      return NV_ERR_CUDA;
    attr_bytes = sm;
  }
  const int sms = num_sms();
  if (sms <= 0) return NV_ERR_CUDA;
  const int64_t ctas = (int64_t)sms * (NACC == 1 ? 2 : 1);  // one accumulator: two CTAs share an SM
  const int64_t grid = max_tiles < ctas ? max_tiles : ctas;
  if (grid <= 0) return NV_OK;
  k<<<(unsigned)grid, 192, sm, s>>>(ta, tb, args);
  return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

template <int KIND, int STAGES, int BN, int CHUNKS = 1, bool kSwb = false>
static int run_pair(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tsa, const CUtensorMap &tsb,
                    const GemmArgs &args, int64_t max_tiles, cudaStream_t s) {
  using C = CfgPair<KIND, STAGES, BN, CHUNKS>;
  const size_t sm = C::smem_bytes(args.E);
  auto k = grouped_gemm_pair_kernel<KIND, STAGES, BN, CHUNKS, kSwb>;
  static size_t attr_bytes = 0;
  static int max_pairs = 0;  // co-resident CTA pairs at the largest shared-memory size requested so far
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (sm > attr_bytes) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess)
      return NV_ERR_CUDA;
    const int sms = num_sms();
    if (sms <= 0) return NV_ERR_CUDA;
    cfg.gridDim = dim3((unsigned)(4 * sms), 1, 1);  // large enough not to cap the answer
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess || n <= 0) return NV_ERR_CUDA;
    // measured: for two CTAs per SM the query reports one pair per SM pair
    // while the GPU runs two at once (the 256 x 128 variant then takes half
    // the time); a persistent grid larger than what fits only queues pairs
    max_pairs = n > (sms / 2) * C::kCtasPerSm ? n : (sms / 2) * C::kCtasPerSm;
    attr_bytes = sm;
  }
  const int64_t pairs = max_tiles < max_pairs ? max_tiles : max_pairs;
  if (pairs <= 0) return NV_OK;
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  if (cudaLaunchKernelEx(&cfg, k, ta, tb, tsa, tsb, args) != cudaSuccess) return NV_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

// Which kernel runs a problem: the CTA-pair kernel needs 256-wide output
// tiles; for fwd and dgrad it pays off only when the experts hold several
// 128-row blocks each (a half-empty pair tile wastes half of its MMAs).
static volatile int g_variant = -1;  // -1: not yet read from the environment

static int gemm_variant() {
  if (g_variant < 0) {
    const char *e = getenv("NVFP4MOE_GEMM_VARIANT");
    const int v = e ? atoi(e) : 0;
    g_variant = (v >= 0 && v <= 4) ? v : 0;
  }
  return g_variant;
}

// Limit of the GEMMs' pipeline waits (polls); the default lets a wait last
// far longer than any healthy step takes.
static volatile uint64_t g_wait_limit = (uint64_t)1 << 26;

int set_gemm_wait_limit(int64_t spins) {
  if (spins < 0 || spins > ((int64_t)1 << 26)) return NV_ERR_ARG;
  g_wait_limit = spins == 0 ? ((uint64_t)1 << 26) : (uint64_t)spins;
  return NV_OK;
}

int set_gemm_variant(int v) {
  if (v < 0 || v > 4) return NV_ERR_ARG;
  g_variant = v;
  return NV_OK;
}

int launch_grouped_gemm(const GemmProblem &p, int *status, cudaStream_t s) {
  if (p.M_total == 0 && p.kind != kGemmMxfp8Dw) return NV_OK;
  const int64_t P = nvfp4moe_padded_cap(p.M_total, p.E);
  GemmArgs a = {};
  a.a_scales = p.a_scales; a.b_scales = p.b_scales; a.a_sg = p.a_sg; a.b_sg = p.b_sg;
  a.groups = p.groups; a.E = p.E; a.M_total = p.M_total; a.N = p.N; a.K = p.K;
  a.out = p.out; a.out_fp32 = p.out_fp32; a.status = status;
  a.wait_limit = g_wait_limit;
  a.h = p.h; a.h_amax = reinterpret_cast<unsigned *>(p.h_amax); a.I = p.N / 2;
  a.a_sg_rows = p.a_sg_rows; a.h_amax_rows = p.h_amax_rows;
  a.s2f6_codes = p.s2f6_codes; a.s2f6_scales = p.s2f6_scales;
  if (p.s2f6_codes) a.rht = make_signs(p.rht_signs);
  a.swb_y13 = p.swb_y13;
  const int64_t out_cols = (p.kind == kGemmNvfp4Fwd || p.kind == kGemmNvfp4FwdSwiglu) ? p.N : p.K;
  CUtensorMap ta, tb;
  bool ok;
  switch (p.kind) {
    case kGemmNvfp4Fwd:
      ok = make_map(&ta, p.a_codes, p.K / 2, p.M_total, p.K / 2, 128) &&
           make_map(&tb, p.b_codes, p.K / 2, (uint64_t)p.E * p.N, p.K / 2, kBN);
      a.ka = p.K / 64;
      break;
    case kGemmNvfp4FwdSwiglu:  // B in boxes of 64 rows: gate rows, then the matching up rows
      ok = make_map(&ta, p.a_codes, p.K / 2, p.M_total, p.K / 2, 128) &&
           make_map(&tb, p.b_codes, p.K / 2, (uint64_t)p.E * p.N, p.K / 2, 64);
      a.ka = p.K / 64;
      break;
    case kGemmMxfp8Dx:
      ok = make_map(&ta, p.a_codes, p.N, p.M_total, p.N, 128) &&
           make_map(&tb, p.b_codes, p.N, (uint64_t)p.E * p.K, p.N, kBN);
      a.ka = p.N / 128;
      break;
    default:
      ok = make_map(&ta, p.a_codes, P, p.N, P, 128) && make_map(&tb, p.b_codes, P, p.K, P, kBN);
      a.ka = P / 128;
      break;
  }
  if (!ok) return NV_ERR_CUDA;
  a.ntn = (int)(out_cols / kBN);
  a.out_ld = out_cols;
  int64_t max_tiles;
  if (p.kind == kGemmMxfp8Dw) {
    a.ntm = (int)(p.N / 128);
    max_tiles = (int64_t)p.E * a.ntm * a.ntn;
  } else {
    max_tiles = (P / 128) * a.ntn;
  }
  // variants: 1 one CTA per SM with two accumulators (6 stages); 2 two CTAs
  // per SM with one accumulator each (3 stages); 3 CTA pairs with 256 x 256
  // tiles; 4 CTA pairs with 256 x 128 tiles, two pairs per SM pair.  A pair
  // variant applies where the shape allows it (else 2).  Automatic: 3 when the
  // experts hold several 128-row blocks (a half-empty pair block wastes half
  // of its MMAs), else 2.  Measured at the MoE shapes (16384 tokens, 64
  // experts, ms, variants 2 / 3): NVFP4 forward w13 0.78 / 0.68, w2 0.48 /
  // 0.42; MXFP8 dgrad and wgrad faster with 3 as well.  The SwiGLU kind has
  // no 256 x 128 pair form (its 64 gate + 64 up rows would split scale tiles).
  if (p.s2f6_codes)  // the RHT + S2F6 epilogue exists in the 128 x 128 kernel only
    return run<kGemmNvfp4Fwd, 3, 1, true>(ta, tb, a, max_tiles, s);
  const int forced = gemm_variant();
  const bool rows_ok = p.kind != kGemmMxfp8Dw || p.N % 256 == 0;  // wgrad: pair tiles of 256 rows
  const bool big_groups = p.kind == kGemmMxfp8Dw || p.M_total >= (int64_t)512 * p.E;
  int pair_bn = 0;
  if (forced == 3 || forced == 4) {
    pair_bn = forced == 3 ? 256 : 128;
  } else if (forced == 0 && big_groups) {
    pair_bn = 256;
  }
  if (pair_bn && (!rows_ok || out_cols % pair_bn)) pair_bn = 0;
  if (p.kind == kGemmNvfp4FwdSwiglu && pair_bn != 256)  // 128 x (64 gate + 64 up), two CTAs per SM
    return run<kGemmNvfp4FwdSwiglu, 3, 1>(ta, tb, a, max_tiles, s);
  if (pair_bn) {
    const int atoms = (p.kind == kGemmNvfp4Fwd || p.kind == kGemmNvfp4FwdSwiglu) ? 4 : 1;
    uint64_t a_sf_bytes, b_sf_bytes;
    switch (p.kind) {
      case kGemmNvfp4Fwd:
      case kGemmNvfp4FwdSwiglu:
        a_sf_bytes = (uint64_t)(P / 128) * a.ka * 512;
        b_sf_bytes = (uint64_t)(p.E * p.N / 128) * a.ka * 512;
        break;
      case kGemmMxfp8Dx:
        a_sf_bytes = (uint64_t)(P / 128) * a.ka * 512;
        b_sf_bytes = (uint64_t)(p.E * p.K / 128) * a.ka * 512;
        break;
      default:
        a_sf_bytes = (uint64_t)(p.N / 128) * a.ka * 512;
        b_sf_bytes = (uint64_t)(p.K / 128) * a.ka * 512;
        break;
    }
    CUtensorMap tsa, tsb, tbh;
    // 256-wide tiles take two B scale tiles per k-atom, one 4-D load
    const uint64_t sf_gap = p.kind == kGemmNvfp4FwdSwiglu ? (uint64_t)(p.N / 2) / 128 : 1;
    if (!make_sf_map(&tsa, p.a_scales, a_sf_bytes, 4 * atoms) ||
        !(pair_bn == 256 ? make_sf_map_pair(&tsb, p.b_scales, b_sf_bytes / (a.ka * 512), a.ka, sf_gap, 4 * atoms)
                         : make_sf_map(&tsb, p.b_scales, b_sf_bytes, 4 * atoms)))
      return NV_ERR_CUDA;
    const CUtensorMap *tbp = &tb;  // B box of BN / 2 rows
    if (p.kind == kGemmNvfp4FwdSwiglu) {  // 128 gate or up rows per CTA
      if (!make_map(&tbh, p.b_codes, p.K / 2, (uint64_t)p.E * p.N, p.K / 2, 128)) return NV_ERR_CUDA;
      tbp = &tbh;
    } else if (pair_bn == 128) {
      switch (p.kind) {
        case kGemmNvfp4Fwd: ok = make_map(&tbh, p.b_codes, p.K / 2, (uint64_t)p.E * p.N, p.K / 2, 64); break;
        case kGemmMxfp8Dx: ok = make_map(&tbh, p.b_codes, p.N, (uint64_t)p.E * p.K, p.N, 64); break;
        default: ok = make_map(&tbh, p.b_codes, P, p.K, P, 64); break;
      }
      if (!ok) return NV_ERR_CUDA;
      tbp = &tbh;
    }
    GemmArgs b = a;
    b.ntn = (int)(out_cols / pair_bn);
    int64_t pair_tiles;
    if (p.kind == kGemmMxfp8Dw) {
      b.ntm = (int)(p.N / 256);
      pair_tiles = (int64_t)p.E * b.ntm * b.ntn;
    } else {
      pair_tiles = ((P / 128 + p.E) / 2) * b.ntn;  // upper bound of sum_e ceil(P_e / 256) tiles
    }
    if (pair_bn == 256 && (p.kind == kGemmMxfp8Dx || p.kind == kGemmMxfp8Dw)) {
      // two-chunk stages with wide loads (see CfgPair::kWideLoads)
      const bool dx = p.kind == kGemmMxfp8Dx;
      const uint64_t row_bytes = dx ? (uint64_t)p.N : (uint64_t)P;
      const uint64_t a_rows = dx ? (uint64_t)p.M_total : (uint64_t)p.N;
      const uint64_t b_rows = dx ? (uint64_t)p.E * p.K : (uint64_t)p.K;
      CUtensorMap wa, wb, wsa, wsb;
      if (!make_map_chunks(&wa, p.a_codes, row_bytes, a_rows, 128) ||
          !make_map_chunks(&wb, p.b_codes, row_bytes, b_rows, 128) || !make_sf_map(&wsa, p.a_scales, a_sf_bytes, 8) ||
          !make_sf_map_pair_chunks(&wsb, p.b_scales, b_sf_bytes / (a.ka * 512), a.ka, 1, 4))
        return NV_ERR_CUDA;
      if (dx && p.swb_y13) return run_pair<kGemmMxfp8Dx, 3, 256, 2, true>(wa, wb, wsa, wsb, b, pair_tiles, s);
      return dx ? run_pair<kGemmMxfp8Dx, 3, 256, 2>(wa, wb, wsa, wsb, b, pair_tiles, s)
                : run_pair<kGemmMxfp8Dw, 3, 256, 2>(wa, wb, wsa, wsb, b, pair_tiles, s);
    }
    if (pair_bn == 256) {
      switch (p.kind) {
        case kGemmNvfp4Fwd: return run_pair<kGemmNvfp4Fwd, 5, 256>(ta, *tbp, tsa, tsb, b, pair_tiles, s);
        case kGemmNvfp4FwdSwiglu:
          return run_pair<kGemmNvfp4FwdSwiglu, 5, 256>(ta, *tbp, tsa, tsb, b, pair_tiles, s);
        case kGemmMxfp8Dx:
          return p.swb_y13 ? run_pair<kGemmMxfp8Dx, 3, 256, 2, true>(ta, *tbp, tsa, tsb, b, pair_tiles, s)
                           : run_pair<kGemmMxfp8Dx, 3, 256, 2>(ta, *tbp, tsa, tsb, b, pair_tiles, s);
        default: return run_pair<kGemmMxfp8Dw, 3, 256, 2>(ta, *tbp, tsa, tsb, b, pair_tiles, s);
      }
    }
    switch (p.kind) {
      case kGemmNvfp4Fwd: return run_pair<kGemmNvfp4Fwd, 3, 128>(ta, *tbp, tsa, tsb, b, pair_tiles, s);
      case kGemmMxfp8Dx:
        return p.swb_y13 ? run_pair<kGemmMxfp8Dx, 4, 128, 1, true>(ta, *tbp, tsa, tsb, b, pair_tiles, s)
                         : run_pair<kGemmMxfp8Dx, 4, 128>(ta, *tbp, tsa, tsb, b, pair_tiles, s);
      default: return run_pair<kGemmMxfp8Dw, 4, 128>(ta, *tbp, tsa, tsb, b, pair_tiles, s);
    }
  }
  const bool two_per_sm = forced != 1;
  switch (p.kind) {
    case kGemmNvfp4Fwd:
      return two_per_sm ? run<kGemmNvfp4Fwd, 3, 1>(ta, tb, a, max_tiles, s)
                        : run<kGemmNvfp4Fwd, 6, 2>(ta, tb, a, max_tiles, s);
    case kGemmMxfp8Dx:
      if (p.swb_y13)
        return two_per_sm ? run<kGemmMxfp8Dx, 3, 1, false, true>(ta, tb, a, max_tiles, s)
                          : run<kGemmMxfp8Dx, 6, 2, false, true>(ta, tb, a, max_tiles, s);
      return two_per_sm ? run<kGemmMxfp8Dx, 3, 1>(ta, tb, a, max_tiles, s)
                        : run<kGemmMxfp8Dx, 6, 2>(ta, tb, a, max_tiles, s);
    default:
      return two_per_sm ? run<kGemmMxfp8Dw, 3, 1>(ta, tb, a, max_tiles, s)
                        : run<kGemmMxfp8Dw, 6, 2>(ta, tb, a, max_tiles, s);
  }
}

}  // namespace nvm
