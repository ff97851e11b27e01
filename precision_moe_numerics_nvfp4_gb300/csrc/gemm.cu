// Grouped block-scaled expert GEMMs on the 5th-generation tensor cores
// (tcgen05), steps a3, a7 and a8 of the hot path:
//   NVFP4 forward   y_e  = x_q,e w_q,e^T      kind::mxf4nvf4, E4M3 scales / 16
//   MXFP8 dgrad     dx_e = g_e w_e            kind::mxf8f6f4, E8M0 scales / 32
//   MXFP8 wgrad     dw_e = g_e^T x_q,e        kind::mxf8f6f4, contraction over
//                                             the expert's padded tokens
// "End-to-End 4-Bit Training", "Block-scaled backward passes": a block-scaled
// dot product multiplies pairs of a 16- (or 32-) value block from each operand,
// sums them and scales the sum by both block scales; "Kernels for
// low-precision training": the MoE layer is dominated by these GEMMs.
//
// One CTA computes one 128 x BN output tile with all of K:
//   warp 0      TMA producer: A/B tiles (128-byte swizzle) and the scale tiles
//               (1-D bulk copies of whole 512-byte 128x4 scale tiles) into a
//               STAGES-deep shared-memory ring, one mbarrier per stage
//   warp 1      allocates tensor memory; one thread copies the stage's scales
//               to tensor memory (tcgen05.cp) and issues 4 block-scaled MMAs
//               per stage into a 128 x BN fp32 accumulator in tensor memory;
//               tcgen05.commit frees the stage
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, outer-scale multiply,
//               bf16/fp32 stores of the rows that belong to the expert
// Every wait is bounded: a wait that runs out records NV_ERR_TIMEOUT, stops
// issuing, waits (bounded) for its own copies, frees tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"

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
__device__ __forceinline__ void mma_mxf8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

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

template <int KIND, int BN, int STAGES>
struct Cfg {
  static constexpr bool kFp4 = KIND == kGemmNvfp4Fwd;
  static constexpr int kAtomsPerStage = kFp4 ? 4 : 1;  // 128x4 scale tiles per 128 rows per stage
  static constexpr int A_BYTES = 128 * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int SFA_BYTES = kAtomsPerStage * 512;
  static constexpr int SFB_BYTES = (BN / 128) * SFA_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int SFA_COLS = kAtomsPerStage * 4;         // tensor-memory columns per stage
  static constexpr int SFB_COLS = kAtomsPerStage * (BN / 32);
  static constexpr int SF_COLS = SFA_COLS + SFB_COLS;
  static constexpr int TMEM_COLS = cpow2(BN + 2 * SF_COLS);
  static constexpr int BAR_BYTES = (2 * STAGES + 1) * 8 + 16;
  static constexpr uint32_t IDESC =
      (kFp4 ? ((1u << 7) | (1u << 10)) : (1u << 23)) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  static size_t smem_bytes(int E) {
    return 1024 + (size_t)STAGES * STAGE_BYTES + BAR_BYTES + (size_t)(E + 1) * 8 + 64;
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
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int KIND, int BN, int STAGES>
__global__ void __launch_bounds__(192, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmArgs A) {
  using C = Cfg<KIND, BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t *sA = smem;
  uint8_t *sB = sA + STAGES * C::A_BYTES;
  uint8_t *sSFA = sB + STAGES * C::B_BYTES;
  uint8_t *sSFB = sSFA + STAGES * C::SFA_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sSFB + STAGES * C::SFB_BYTES);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 1);
  int *s_flag = reinterpret_cast<int *>(s_tmem + 2);
  int *s_off = s_flag + 2;
  int *s_pad = s_off + (A.E + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!load_groups(A.groups, A.E, A.M_total, s_off, s_pad, s_flag, A.status)) return;

  // ---- which tile -----------------------------------------------------------
  int e, nk, a_row, b_row, mrows, k_off;
  int64_t a_tile, b_tile, k_atom0, out_row0, out_col0;
  if (KIND != kGemmMxfp8Dw) {
    const int pm = blockIdx.x / A.ntn, nt = blockIdx.x - (blockIdx.x / A.ntn) * A.ntn;
    const int p0 = pm * 128;
    if (p0 >= s_pad[A.E]) return;  // past the last group (uniform over the CTA)
    e = find_group(s_pad, A.E, p0);
    a_row = s_off[e] + (p0 - s_pad[e]);
    mrows = min(128, s_off[e + 1] - a_row);
    b_row = e * (int)(KIND == kGemmNvfp4Fwd ? A.N : A.K) + nt * BN;
    a_tile = pm;
    b_tile = b_row / 128;
    nk = (int)(KIND == kGemmNvfp4Fwd ? A.K / 256 : A.N / 128);
    k_off = 0;
    k_atom0 = 0;
    out_row0 = a_row;
    out_col0 = (int64_t)nt * BN;
  } else {
    const int per_e = A.ntm * A.ntn;
    e = blockIdx.x / per_e;
    const int r = blockIdx.x - e * per_e, mt = r / A.ntn, nt = r - (r / A.ntn) * A.ntn;
    a_row = mt * 128;
    b_row = nt * BN;
    mrows = 128;
    nk = (s_pad[e + 1] - s_pad[e]) / 128;
    k_off = s_pad[e];
    a_tile = mt;
    b_tile = b_row / 128;
    k_atom0 = s_pad[e] / 128;
    out_row0 = (int64_t)e * A.N + (int64_t)mt * 128;
    out_col0 = (int64_t)nt * BN;
  }

  uint64_t *full = bars, *empty = bars + STAGES, *accb = bars + 2 * STAGES;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(accb), 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(s_tmem), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 0 && lane == 0) {
    // ---- producer -----------------------------------------------------------
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
    int issued = 0;
    for (int ks = 0; ks < nk; ++ks) {
      const int s = ks % STAGES;
      if (ks >= STAGES && !mbar_wait(smem_u32(&empty[s]), ((ks / STAGES) - 1) & 1, A.wait_limit)) {
        record_error(A.status, NV_ERR_TIMEOUT);
        break;
      }
      const uint32_t fb = smem_u32(&full[s]);
      mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
      tma_load_2d(smem_u32(sA + s * C::A_BYTES), &tmA, k_off + ks * 128, a_row, fb);
      tma_load_2d(smem_u32(sB + s * C::B_BYTES), &tmB, k_off + ks * 128, b_row, fb);
      const int64_t katom = k_atom0 + (int64_t)ks * C::kAtomsPerStage;
      bulk_load(smem_u32(sSFA + s * C::SFA_BYTES), A.a_scales + (a_tile * A.ka + katom) * 512, C::SFA_BYTES, fb);
#pragma unroll
      for (int j = 0; j < BN / 128; ++j)
        bulk_load(smem_u32(sSFB + s * C::SFB_BYTES + j * C::SFA_BYTES),
                  A.b_scales + ((b_tile + j) * A.ka + katom) * 512, C::SFA_BYTES, fb);
      issued = ks + 1;
    }
    // drain: every copy this thread issued has landed before the CTA leaves
    for (int ks = issued > STAGES ? issued - STAGES : 0; ks < issued; ++ks)
      if (!mbar_wait(smem_u32(&full[ks % STAGES]), (ks / STAGES) & 1, A.wait_limit)) {
        record_error(A.status, NV_ERR_TIMEOUT);
        break;
      }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ------------------------------------------------------------
    for (int ks = 0; ks < nk; ++ks) {
      const int s = ks % STAGES;
      if (!mbar_wait(smem_u32(&full[s]), (ks / STAGES) & 1, A.wait_limit)) {
        record_error(A.status, NV_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      // the scale buffer about to be overwritten was last read by stage ks-2
      if (ks >= 2 && !mbar_wait(smem_u32(&empty[(ks - 2) % STAGES]), ((ks - 2) / STAGES) & 1, A.wait_limit)) {
        record_error(A.status, NV_ERR_TIMEOUT);
        break;
      }
      const uint32_t sfa = tmem + BN + (ks & 1) * C::SF_COLS;
      const uint32_t sfb = sfa + C::SFA_COLS;
      const uint32_t a_sf_smem = smem_u32(sSFA + s * C::SFA_BYTES);
      const uint32_t b_sf_smem = smem_u32(sSFB + s * C::SFB_BYTES);
#pragma unroll
      for (int j = 0; j < C::kAtomsPerStage; ++j) {
        tc_cp_sf(sfa + 4 * j, desc_sf(a_sf_smem + j * 512));
#pragma unroll
        for (int r = 0; r < BN / 128; ++r)
          tc_cp_sf(sfb + j * (BN / 32) + 4 * r, desc_sf(b_sf_smem + r * C::SFA_BYTES + j * 512));
      }
      const uint64_t da = desc_sw128(smem_u32(sA + s * C::A_BYTES));
      const uint64_t db = desc_sw128(smem_u32(sB + s * C::B_BYTES));
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t acc = (ks | j) != 0;
        if (C::kFp4) {
          mma_nvf4(tmem, da + 2 * j, db + 2 * j, C::IDESC, sfa + 4 * j, sfb + j * (BN / 32), acc);
        } else {
          const uint32_t idesc = C::IDESC | ((uint32_t)j << 4) | ((uint32_t)j << 29);
          mma_mxf8(tmem, da + 2 * j, db + 2 * j, idesc, sfa, sfb, acc);
        }
      }
      tc_commit(smem_u32(&empty[s]));
    }
    tc_commit(smem_u32(accb));
  } else if (warp >= 2) {
    // ---- epilogue ----------------------------------------------------------------
    const int q = warp & 3;
    const int row = q * 32 + lane;
    bool ok = true;
    if (nk > 0) {
      ok = mbar_wait(smem_u32(accb), 0, A.wait_limit);
      if (!ok) record_error(A.status, NV_ERR_TIMEOUT);
      tc_fence_after();
    }
    if (ok) {
      float alpha = 1.0f;
      if (KIND == kGemmNvfp4Fwd) alpha = __fmul_rn(A.a_sg[0], A.b_sg[e]);
      const bool store = row < mrows;
      const int64_t orow = out_row0 + row;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        if (nk > 0) {
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (!store) continue;
        if (A.out_fp32) {
          float *dst = static_cast<float *>(A.out) + orow * A.out_ld + out_col0 + c0;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4 *>(dst + i) =
                make_float4(__fmul_rn(__uint_as_float(v[i]), alpha), __fmul_rn(__uint_as_float(v[i + 1]), alpha),
                            __fmul_rn(__uint_as_float(v[i + 2]), alpha), __fmul_rn(__uint_as_float(v[i + 3]), alpha));
        } else {
          uint16_t *dst = static_cast<uint16_t *>(A.out) + orow * A.out_ld + out_col0 + c0;
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            w.x = pack_bf16x2(__fmul_rn(__uint_as_float(v[i]), alpha), __fmul_rn(__uint_as_float(v[i + 1]), alpha));
            w.y = pack_bf16x2(__fmul_rn(__uint_as_float(v[i + 2]), alpha), __fmul_rn(__uint_as_float(v[i + 3]), alpha));
            w.z = pack_bf16x2(__fmul_rn(__uint_as_float(v[i + 4]), alpha), __fmul_rn(__uint_as_float(v[i + 5]), alpha));
            w.w = pack_bf16x2(__fmul_rn(__uint_as_float(v[i + 6]), alpha), __fmul_rn(__uint_as_float(v[i + 7]), alpha));
            *reinterpret_cast<uint4 *>(dst + i) = w;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
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

template <int KIND, int BN, int STAGES>
static int run(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &args, int64_t grid, cudaStream_t s) {
  using C = Cfg<KIND, BN, STAGES>;
  const size_t sm = C::smem_bytes(args.E);
  auto k = grouped_gemm_kernel<KIND, BN, STAGES>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess) return NV_ERR_CUDA;
  if (grid <= 0) return NV_OK;
  k<<<(unsigned)grid, 192, sm, s>>>(ta, tb, args);
  return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

int launch_grouped_gemm(const GemmProblem &p, int *status, cudaStream_t s) {
  if (p.M_total == 0 && p.kind != kGemmMxfp8Dw) return NV_OK;
  const int64_t P = nvfp4moe_padded_cap(p.M_total, p.E);
  GemmArgs a = {};
  a.a_scales = p.a_scales; a.b_scales = p.b_scales; a.a_sg = p.a_sg; a.b_sg = p.b_sg;
  a.groups = p.groups; a.E = p.E; a.M_total = p.M_total; a.N = p.N; a.K = p.K;
  a.out = p.out; a.out_fp32 = p.out_fp32; a.status = status;
  a.wait_limit = (uint64_t)1 << 26;
  CUtensorMap ta, tb;
  const int bn = 256;
  int64_t out_cols, grid;
  bool ok;
  switch (p.kind) {
    case kGemmNvfp4Fwd:
      out_cols = p.N;
      ok = make_map(&ta, p.a_codes, p.K / 2, p.M_total, p.K / 2, 128) &&
           make_map(&tb, p.b_codes, p.K / 2, (uint64_t)p.E * p.N, p.K / 2, (out_cols % bn) ? 128 : bn);
      a.ka = p.K / 64;
      break;
    case kGemmMxfp8Dx:
      out_cols = p.K;
      ok = make_map(&ta, p.a_codes, p.N, p.M_total, p.N, 128) &&
           make_map(&tb, p.b_codes, p.N, (uint64_t)p.E * p.K, p.N, (out_cols % bn) ? 128 : bn);
      a.ka = p.N / 128;
      break;
    default:
      out_cols = p.K;
      ok = make_map(&ta, p.a_codes, P, p.N, P, 128) && make_map(&tb, p.b_codes, P, p.K, P, (out_cols % bn) ? 128 : bn);
      a.ka = P / 128;
      break;
  }
  if (!ok) return NV_ERR_CUDA;
  const bool wide = out_cols % bn == 0;
  a.ntn = (int)(out_cols / (wide ? 256 : 128));
  a.out_ld = out_cols;
  if (p.kind == kGemmMxfp8Dw) {
    a.ntm = (int)(p.N / 128);
    grid = (int64_t)p.E * a.ntm * a.ntn;
  } else {
    grid = (P / 128) * a.ntn;
  }
  switch (p.kind) {
    case kGemmNvfp4Fwd:
      return wide ? run<kGemmNvfp4Fwd, 256, 4>(ta, tb, a, grid, s) : run<kGemmNvfp4Fwd, 128, 5>(ta, tb, a, grid, s);
    case kGemmMxfp8Dx:
      return wide ? run<kGemmMxfp8Dx, 256, 4>(ta, tb, a, grid, s) : run<kGemmMxfp8Dx, 128, 6>(ta, tb, a, grid, s);
    default:
      return wide ? run<kGemmMxfp8Dw, 256, 4>(ta, tb, a, grid, s) : run<kGemmMxfp8Dw, 128, 6>(ta, tb, a, grid, s);
  }
}

}  // namespace nvm
