/*
 * nvfp4moe.h -- C ABI of libnvfp4moe.so: the data-parallel hot path of
 * NVFP4-forward / MXFP8-backward MoE expert training on one GB300 (sm_103a).
 *
 * The method is the one described in "End-to-End 4-Bit Training" (Thinking
 * Machines Lab): NVFP4 block quantization of activations and weights, grouped
 * NVFP4 expert GEMMs in the forward pass, dequantize -> transpose -> stochastic
 * re-quantization of the saved forward tensors to MXFP8, SR quantization of
 * the BF16 output gradient, and grouped MXFP8 dgrad / wgrad GEMMs.
 *
 * General rules (every entry point):
 *  - Pointers are DEVICE pointers unless a parameter says otherwise.  The
 *    caller owns and allocates every buffer, including workspaces; the library
 *    never allocates or frees device memory.  Its only device memory of its
 *    own is the status word and the fixed scratch of nvfp4_quantize_noalloc.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream) and is asynchronous.  The return value reports argument checks
 *    and launch errors only (NV_OK or a negative NV_ERR_*).  Errors the GPU
 *    detects (inconsistent group offsets, a bounded wait that ran out) are
 *    recorded in a per-device status word read by nvfp4moe_get_device_status.
 *    No kernel traps or prints.
 *  - Every pointer must be 16-byte aligned.  Results are bitwise
 *    deterministic: the same inputs give the same bytes on every run.
 *  - Matrices are row-major.  bf16 is IEEE bfloat16 bits (uint16).
 *
 * Number formats ("Low-precision formats on Blackwell" on the pages):
 *  - E2M1 (FP4): +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}; two per byte, element 2j in
 *    the low nibble of byte j.
 *  - E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; largest 448; used for
 *    NVFP4 block scales and for MXFP8 elements.
 *  - E8M0: 2^(code - 127); MXFP8 block scales.
 *  - NVFP4: E2M1 codes, one E4M3 scale per 16 consecutive values of a row and
 *    one FP32 outer scale per tensor: x = e2m1 * e4m3 * sg.
 *  - MXFP8: E4M3 codes, one E8M0 scale per 32 consecutive values of a row.
 *
 * Conventions the pages leave open (identical in the CPU oracle):
 *  - sg = amax / (6 * 448) per tensor (per expert matrix for weights), 1 for
 *    an all-zero tensor; NVFP4 scale s = RN_E4M3(blockamax / (6 * sg))
 *    saturating at 448; codes = RN_E2M1(x * (1 / (s * sg))); an all-zero (or
 *    underflowed) block gets scale 0 and signed-zero codes.  All steps are
 *    IEEE fp32, round to nearest even.
 *  - MXFP8 scale = floor(log2 blockamax) - 8 clamped to [-127, 127] (OCP MX),
 *    code = scale + 127; scale code 0 and signed zeros for an all-zero block;
 *    elements RN or SR to E4M3 saturating at 448.
 *  - Stochastic rounding ("Re-quantization with stochastic rounding"): with
 *    a <= |w| < b the neighbouring E4M3 values, round up iff
 *    r < floor(2^16 (|w| - a) / (b - a)), r = a 16-bit draw.  (This is the
 *    rule of Blackwell's hardware SR conversion, which the kernels use.)
 *  - Draws: one 16-bit draw U per PAIR of output elements (two consecutive
 *    elements along the output row / MXFP8 block); the first element uses U,
 *    the second bitrev16(U).  U(K) is the 16-bit half (K & 1) of word
 *    (K >> 1) & 3 of Philox4x32-10 (Salmon et al., SC'11) with key = (seed lo,
 *    seed hi) and counter = (q lo, q hi, offset lo, offset hi), q = K >> 3.
 *    The pair key K comes from the source position (r, c) of the pair's first
 *    element in a source with C columns: K = (r * C + c) / 2 for row-wise
 *    outputs (pairs of columns), K = r * C + c for transposed outputs (pairs
 *    of rows).  For stacked weights r is the row in the [batch * rows] stack.
 *
 * Scale-factor layout (all block scales, NVFP4 and MXFP8): the 128x4 tile
 * that block-scaled tcgen05 MMA reads.  The scale of padded row r', block
 * column c, in a matrix with KB block columns is at byte
 *     ((r' / 128) * ceil(KB / 4) + c / 4) * 512 + (r' % 32) * 16
 *       + ((r' / 32) % 4) * 4 + c % 4,
 * every padding byte zero.  Padded rows: a stack of `batch` matrices with R
 * rows uses r' = b * roundup(R, 128) + r; a matrix whose rows are grouped by
 * expert (group_offsets o, sizes M_e = o[e+1] - o[e]) uses
 * r' = P_e + (r - o[e]) with P_e = sum_{e' < e} roundup(M_e', 128), so that
 * every 128-row tile of an expert owns its scale atoms.  Grouped buffers are
 * sized for P_cap = nvfp4moe_padded_cap(M_total, E) rows.
 *
 * group_offsets: int32 [E + 1] on the device, 1 <= E <= 512, o[0] = 0,
 * non-decreasing, o[E] = M_total.  Empty groups are allowed.  Kernels that read them record
 * NV_ERR_OFFSETS in the status word (and write nothing) when they are
 * inconsistent.
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *nv_stream_t; /* a cudaStream_t */

enum nv_status {
  NV_OK = 0,
  NV_ERR_ARG = -1,          /* null pointer, negative size, bad enum */
  NV_ERR_ALIGN = -2,        /* a pointer is not 16-byte aligned */
  NV_ERR_SHAPE = -3,        /* a size violates the divisibility rules */
  NV_ERR_OFFSETS = -4,      /* (device) group offsets inconsistent */
  NV_ERR_TIMEOUT = -5,      /* (device) a bounded wait ran out */
  NV_ERR_CUDA = -6,         /* a CUDA runtime call failed */
  NV_ERR_UNSUPPORTED = -7,  /* a feature or GPU the compiled library does not support */
  NV_ERR_WORKSPACE = -8     /* workspace missing or too small */
};
enum nv_round { NV_RN = 0, NV_SR = 1 };
enum nv_out_dtype { NV_OUT_BF16 = 0, NV_OUT_FP32 = 1 };

/* ---- sizes and layout helpers (host only, no GPU work) --------------------- */

/* Padded rows reserved for a grouped layout: roundup(M_total + 127 E, 128). */
int64_t nvfp4moe_padded_cap(int64_t M_total, int64_t E);

/* Bytes of a scale buffer for `padded_rows` rows and `kblocks` block columns:
 * roundup(padded_rows, 128) / 128 * ceil(kblocks / 4) * 512. */
int64_t nvfp4moe_scale_bytes(int64_t padded_rows, int64_t kblocks);

/* Byte offset of the scale of padded row rp, block column c (see above). */
int64_t nvfp4moe_scale_offset(int64_t rp, int64_t c, int64_t kblocks);

/* Workspace bytes nvfp4_quantize needs when it computes the outer scales. */
size_t nvfp4moe_quantize_workspace_bytes(int64_t batch, int64_t rows, int64_t cols);

/* Workspace bytes nvfp4_quantize_requant_gather needs: src_rows token rows
 * gathered into rows x cols (the amax pass's scratch and, when src_rows <=
 * rows, the tokens' NVFP4 codes and scales).  0 for negative sizes. */
size_t nvfp4moe_quantize_gather_workspace_bytes(int64_t src_rows, int64_t rows, int64_t cols);

/* Workspace bytes grouped_gemm_nvfp4_fwd needs when it is given bf16
 * activations (x_bf16 non-NULL): their NVFP4 codes, grouped scales, outer
 * scale and the amax pass's scratch.  0 for invalid sizes. */
size_t nvfp4moe_fwd_workspace_bytes(int64_t M_total, int64_t K, int64_t E);

/* ---- NVFP4 quantization (amax -> outer scale, 1x16 RN) ----------------------------------------------
 * "Low-precision formats on Blackwell": block scaling by the largest value of
 * each 16 consecutive values, E4M3 block scale, FP32 outer scale per tensor;
 * "Recipe details": one outer scale per expert for weights.
 *
 * x:        bf16 [batch][rows][cols], cols % 16 == 0.
 * group_offsets / num_groups: NULL / 0 for plain or batched matrices; else
 *           (batch == 1 only) the expert groups of the rows, which selects the
 *           grouped scale layout.
 * outer_scale_in: NULL -> compute sg = amax / 2688 of every batch entry
 *           (the amax pass, one extra read of x) and write it to outer_scale_out
 *           [batch]; non-NULL -> fp32 [batch] scales to use (copied to
 *           outer_scale_out when that is non-NULL).
 * codes:    u8 [batch][rows][cols / 2].
 * scales:   u8, batched layout (batch * roundup(rows,128) padded rows) or
 *           grouped layout (P_cap padded rows), cols / 16 block columns.
 *           Every byte of the buffer is written (padding zero).
 * workspace: nvfp4moe_quantize_workspace_bytes(...) bytes when
 *           outer_scale_in is NULL, else may be NULL.
 */
int nvfp4_quantize(const void *x, int64_t batch, int64_t rows, int64_t cols,
                   const int32_t *group_offsets, int32_t num_groups,
                   const float *outer_scale_in, float *outer_scale_out,
                   uint8_t *codes, uint8_t *scales,
                   void *workspace, size_t workspace_bytes, nv_stream_t stream);

/* ---- the outer scales alone (the amax pass of nvfp4_quantize) ------------------------
 * sg[b] = amax / 2688 of each of `batch` consecutive bf16 tensors of n values
 * (1 for an all-zero or empty tensor), exactly as nvfp4_quantize computes
 * them; feeding them back as outer_scale_in gives nvfp4_quantize's own
 * result.  Lets the amax pass of one tensor run on another stream while an
 * earlier tensor is being quantized.  n % 8 == 0; x 16-byte aligned;
 * outer_scale_out fp32 [batch]; workspace nvfp4moe_quantize_workspace_bytes(
 * batch, 1, n) bytes (16-byte aligned; else NV_ERR_WORKSPACE).
 */
int nvfp4_outer_scale(const void *x, int64_t batch, int64_t n, float *outer_scale_out,
                      void *workspace, size_t workspace_bytes, nv_stream_t stream);

/* ---- nvfp4_quantize_requant of gathered rows (the expert dispatch) ------------
 * The MoE layer's activations arrive per token; the experts see them per
 * routed row, each token repeated once per expert it is routed to.  This
 * call quantizes the routed-row matrix X without materializing it: row r of
 * X is row row_src[r] of x.  Its outputs are exactly those of
 * nvfp4_quantize_requant on X (the same codes, scales, outer scale and SR
 * draws: draws are keyed by the row of X), for the grouped (expert) layout
 * and the per-tensor outer scale.
 * x:        bf16 [src_rows][cols] (the tokens), cols % 128 == 0.
 * row_src:  int32 [rows] (4-byte aligned), each in [0, src_rows); an index
 *           outside that range makes its row read as zeros and records
 *           NV_ERR_ARG in the device status word.
 * The other arguments as for nvfp4_quantize_requant with batch = 1 and
 * group_offsets required (num_groups >= 1).  The amax pass (outer_scale_in ==
 * NULL) takes the maximum over the rows of X; when src_rows <= rows it reads
 * each token row once (its row maximum) and takes the maximum of those over
 * row_src, the same value.  When src_rows <= rows the tokens are also
 * NVFP4-quantized once, into the workspace, and each routed row's codes and
 * scales are copied from its token's and re-quantized from them (the block
 * rule reads one row at a time, so these are the codes of X's row; a token no
 * row routes may saturate, and is never read).  Workspace:
 * nvfp4moe_quantize_gather_workspace_bytes(src_rows, rows, cols) bytes,
 * 16-byte aligned, required when outer_scale_in is NULL or src_rows <= rows
 * (else NV_ERR_WORKSPACE); otherwise it may be NULL. */
int nvfp4_quantize_requant_gather(const void *x, const int32_t *row_src, int64_t src_rows, int64_t rows,
                                  int64_t cols, const int32_t *group_offsets, int32_t num_groups,
                                  const float *outer_scale_in, float *outer_scale_out, uint8_t *codes,
                                  uint8_t *scales, void *workspace, size_t workspace_bytes, uint64_t seed,
                                  uint64_t counter_offset, uint8_t *out_codes, uint8_t *out_scales,
                                  nv_stream_t stream);

/* ---- nvfp4_quantize for callers that cannot allocate device memory -------------
 * The pages have no counterpart to this entry point; it is a convenience of
 * this library.  nvfp4_quantize needs a caller-provided workspace when it
 * computes the outer scales.  Callers that cannot allocate device memory (code
 * running inside a host runtime that owns every allocation, or that must not
 * allocate once it is running) use this variant, which takes the same
 * arguments minus the workspace and uses a fixed 512 KiB scratch array in the
 * library's own device memory instead.  Every GPU that loads the library
 * holds that array until the process exits.
 *  - Limit: with outer_scale_in == NULL the call needs
 *    nvfp4moe_quantize_workspace_bytes(batch, rows, cols) <= 524288, else it
 *    returns NV_ERR_WORKSPACE and enqueues nothing.  With outer_scale_in set
 *    no scratch is used and there is no limit.
 *  - Arguments are checked exactly as nvfp4_quantize checks them, before the
 *    limit, so a bad call returns the same error through both entry points.
 *  - The first call on a device looks up the scratch's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture.  cudaDeviceReset invalidates the cached addresses (of
 *    this scratch and of the status word): do not call the library again in a
 *    process after resetting a device it has used.
 *  - Every call shares the one array and it keeps the last call's contents;
 *    nothing in it needs clearing (each call writes every slot it reads), but
 *    calls that overlap on the GPU (different streams, or another thread)
 *    race on it: serialize them.
 *  - It calls no cudaMalloc, cudaFree or allocating library routine.
 */
int nvfp4_quantize_noalloc(const void *x, int64_t batch, int64_t rows, int64_t cols,
                           const int32_t *group_offsets, int32_t num_groups,
                           const float *outer_scale_in, float *outer_scale_out,
                           uint8_t *codes, uint8_t *scales, nv_stream_t stream);

/* ---- MXFP8 quantization of a bf16 matrix (the gradient, SR or RN) --------
 * Chinese translation of the pages, Figure 4: the BF16 gradient is quantized
 * to MXFP8 with SR once row-wise (DGRAD operand) and once after a transpose
 * (WGRAD operand).
 *
 * x:        bf16 [rows][cols], cols % 32 == 0.
 * group_offsets / num_groups: expert groups of the rows (NULL / 0: one group
 *           of all rows).
 * mode:     NV_RN or NV_SR; SR draws with (seed, counter_offset_row) for
 *           the row-wise output and (seed, counter_offset_t) for the
 *           transposed one (pair keys as above).
 * codes_row [rows][cols] E4M3, scales_row grouped layout (cols / 32 block
 *           columns; P_cap padded rows, or roundup(rows,128) for one group):
 *           the row-wise output, or both NULL to skip it.
 * codes_t   [cols][P_cap] E4M3: the transpose of each group, zero-padded to
 *           a multiple of 128 tokens and placed at column P_e; blocks of 32
 *           along the new rows.  scales_t: batched layout of one matrix with
 *           `cols` rows and P_cap / 32 block columns.  Columns >= P_total are
 *           left untouched.  Both NULL to skip.  rows with num_groups == 0 are
 *           one group (P_cap = roundup(rows, 128)).
 */
int mxfp8_quantize(const void *x, int64_t rows, int64_t cols,
                   const int32_t *group_offsets, int32_t num_groups,
                   int mode, uint64_t seed, uint64_t counter_offset_row,
                   uint64_t counter_offset_t,
                   uint8_t *codes_row, uint8_t *scales_row,
                   uint8_t *codes_t, uint8_t *scales_t, nv_stream_t stream);

/* ---- dequantize -> transpose -> SR re-quantize NVFP4 -> MXFP8 -------------
 * "Re-quantization with stochastic rounding": the forward NVFP4 tensor is
 * dequantized (fp32: fp32(e2m1 * e4m3) * sg), transposed at that precision,
 * and re-quantized to MXFP8 with stochastic rounding, so that the backward
 * operand equals the forward one in expectation.
 *
 * codes / scales / outer_scale: an nvfp4_quantize output (same batch, rows,
 *           cols, group_offsets); outer_scale fp32 [batch] on the device.
 * Batched (group_offsets NULL): rows % 128 == 0; out_codes [batch][cols][rows]
 *           E4M3, out_scales batched layout (batch matrices of `cols` rows,
 *           rows / 32 block columns).
 * Grouped (batch == 1): out_codes [cols][P_cap] and out_scales as codes_t /
 *           scales_t of mxfp8_quantize.
 * Pair keys for the draws: (b * rows + r0) * cols + c for the pair of
 *           source rows (r0, r0 + 1) of output row c.
 */
int dequant_transpose_requant_sr(const uint8_t *codes, const uint8_t *scales,
                                 const float *outer_scale,
                                 int64_t batch, int64_t rows, int64_t cols,
                                 const int32_t *group_offsets, int32_t num_groups,
                                 uint64_t seed, uint64_t counter_offset,
                                 uint8_t *out_codes, uint8_t *out_scales,
                                 nv_stream_t stream);

/* ---- NVFP4 quantize and the SR re-quantization in one pass ----------
 * Both outputs of nvfp4_quantize (codes, scales, outer scale) and of
 * dequant_transpose_requant_sr applied to them (same seed and counter
 * offset), bit-identical to the two calls in sequence, from one read of the
 * bf16 source: each 128 x 128 tile is quantized to NVFP4 with the block rule
 * of nvfp4_quantize, and the exact products e2m1 * e4m3 of the codes just
 * made feed the transposed stochastic rounding.  For a training step this
 * produces the backward's MXFP8 operand already in the forward pass.
 * No counterpart on the pages as a single operation (a fusion of the two).
 *
 * Arguments: those of nvfp4_quantize, then seed, counter_offset, out_codes,
 * out_scales of dequant_transpose_requant_sr (its layouts).  cols % 128 == 0;
 * batched (group_offsets NULL): rows % 128 == 0.  With outer_scale_in NULL
 * the amax pass runs first (workspace as nvfp4_quantize).
 */
int nvfp4_quantize_requant(const void *x, int64_t batch, int64_t rows, int64_t cols,
                           const int32_t *group_offsets, int32_t num_groups,
                           const float *outer_scale_in, float *outer_scale_out,
                           uint8_t *codes, uint8_t *scales,
                           void *workspace, size_t workspace_bytes,
                           uint64_t seed, uint64_t counter_offset,
                           uint8_t *out_codes, uint8_t *out_scales, nv_stream_t stream);

/* ---- grouped NVFP4 forward GEMM  y_e = x_q,e w_q,e^T ----------------------
 * "Block-scaled backward passes": y = x_q w_q^T, 16-value blocks of a row of
 * x_q and of w_q multiplied pairwise and scaled by both block scales; the
 * outer scales multiply the result (y = acc * sg_x * sg_w[e]).
 *
 * x_codes [M_total][K/2], x_scales grouped layout (K/16 block columns),
 * x_outer_scale fp32 [1]; w_codes [E][N][K/2], w_scales batched layout,
 * w_outer_scale fp32 [E]; y [M_total][N] bf16 or fp32.
 * N % 128 == 0, K % 256 == 0; y 32-byte aligned (the kernels store 32 bytes
 * at a time).
 * x_bf16: NULL -> x_codes / x_scales / x_outer_scale are the quantized
 *   activations and workspace may be NULL.  Non-NULL -> bf16 [M_total][K]
 *   activations (16-byte aligned) that the call quantizes itself exactly as
 *   nvfp4_quantize does (grouped layout; x_outer_scale given, or NULL to
 *   compute it), into the workspace (nvfp4moe_fwd_workspace_bytes(M_total, K,
 *   E) bytes, 16-byte aligned; too small -> NV_ERR_WORKSPACE), before the
 *   GEMM; x_codes / x_scales are ignored.  Bit-identical to the two calls.
 *   (Two passes, not a quantizer inside the GEMM's producer: re-quantizing
 *   each A tile once per N tile costs more than the tile's MMAs here.)
 */
int grouped_gemm_nvfp4_fwd(const void *x_bf16, const float *x_outer_scale,
                           const uint8_t *x_codes, const uint8_t *x_scales,
                           const uint8_t *w_codes, const uint8_t *w_scales,
                           const float *w_outer_scale,
                           const int32_t *group_offsets, int32_t E,
                           int64_t M_total, int64_t N, int64_t K,
                           void *y, int y_dtype,
                           void *workspace, size_t workspace_bytes, nv_stream_t stream);

/* ---- fused: the w13 forward GEMM with SwiGLU in its epilogue ----------
 * Chinese translation, Figure 5 (w13 GEMM -> Q -> w2 GEMM): the gate/up GEMM
 * of grouped_gemm_nvfp4_fwd (bf16 output) on w13 = [E][2I][K] (gate rows
 * 0..I-1 over up rows I..2I-1), and in the same kernel
 *   y13 [M_total][2I] bf16  (bit-identical to grouped_gemm_nvfp4_fwd with
 *                            NV_OUT_BF16),
 *   h   [M_total][I]   bf16  (bit-identical to nvfp4moe_swiglu_fwd of y13),
 *   h_outer_scale [1] fp32   (max |h| / 2688, or 1 when h is all zero:
 *                            bit-identical to the outer scale nvfp4_quantize
 *                            computes for h, so the quantization of h can take
 *                            it as outer_scale_in and skip its amax pass).
 * Each output tile holds 64 hidden features' gate and up columns; max |h| is
 * reduced with atomic max (order-free, deterministic).
 * I % 128 == 0, K % 256 == 0; y13 and h 32-byte aligned.  Other arguments as
 * grouped_gemm_nvfp4_fwd.  No counterpart on the pages as one kernel.
 */
int grouped_gemm_nvfp4_fwd_swiglu(const float *x_outer_scale,
                                  const uint8_t *x_codes, const uint8_t *x_scales,
                                  const uint8_t *w13_codes, const uint8_t *w13_scales,
                                  const float *w13_outer_scale,
                                  const int32_t *group_offsets, int32_t E,
                                  int64_t M_total, int64_t I, int64_t K,
                                  void *y13, void *h, float *h_outer_scale, nv_stream_t stream);

/* ---- grouped MXFP8 dgrad  dx_e = g_e w_e -----------------------------------
 * "Block-scaled backward passes": dx = g w_q, here with both operands MXFP8.
 * g_codes [M_total][N] + g_scales (mxfp8_quantize row-wise output, grouped
 * layout); wt_codes [E][K][N] + wt_scales (dequant_transpose_requant_sr of the
 * weights [E][N][K]); dx [M_total][K] bf16 or fp32, 32-byte aligned.
 * N % 128 == 0, K % 128 == 0.
 */
int grouped_gemm_mxfp8_dx(const uint8_t *g_codes, const uint8_t *g_scales,
                          const uint8_t *wt_codes, const uint8_t *wt_scales,
                          const int32_t *group_offsets, int32_t E,
                          int64_t M_total, int64_t N, int64_t K,
                          void *dx, int dx_dtype,
                          void *workspace, size_t workspace_bytes, nv_stream_t stream);

/* ---- grouped MXFP8 dgrad of the down projection with the SwiGLU backward ------
 * "Block-scaled backward passes" (dh = g2 w2, the dgrad of the down
 * projection) followed by the SwiGLU backward ("MoE expert layer": h =
 * silu(gate) * up), in the GEMM's epilogue: each output dh is rounded to bf16
 * exactly as grouped_gemm_mxfp8_dx writes it, and with the row's gate g and up
 * u of y13, s = sigmoid(g), dgate = dh u s (1 + g (1 - s)) and dup = dh g s
 * are computed in fp32 as nvfp4moe_swiglu_bwd computes them.  The output is
 * exactly grouped_gemm_mxfp8_dx (bf16) followed by nvfp4moe_swiglu_bwd,
 * without dh in memory.  No counterpart on the pages as one kernel.
 * g_codes, g_scales, wt_codes, wt_scales, group_offsets, E, M_total, N as
 * grouped_gemm_mxfp8_dx, with I (its K) the hidden width; y13 [M_total][2I]
 * bf16 (gate columns, then up), read; dy13 [M_total][2I] bf16 (dgate, then
 * dup), written; both 32-byte aligned, not overlapping (else NV_ERR_ARG).
 * N % 128 == 0, I % 128 == 0.
 */
int grouped_gemm_mxfp8_dx_swiglu_bwd(const uint8_t *g_codes, const uint8_t *g_scales,
                                     const uint8_t *wt_codes, const uint8_t *wt_scales,
                                     const int32_t *group_offsets, int32_t E,
                                     int64_t M_total, int64_t N, int64_t I,
                                     const void *y13, void *dy13, nv_stream_t stream);

/* ---- grouped MXFP8 wgrad  dw_e = g_e^T x_q,e ---------------------------------
 * "Block-scaled backward passes": dw = g^T x_q, computed from the quantized
 * forward activations ("Quantized communications": the WGRAD input is the
 * quantized, not the high-precision, activation).  The contraction runs over
 * the tokens of expert e, zero-padded to a multiple of 128.
 * gt_codes [N][P_cap] + gt_scales (mxfp8_quantize transposed output of g),
 * xt_codes [K][P_cap] + xt_scales (dequant_transpose_requant_sr of x_q);
 * dw [E][N][K] fp32 (experts without tokens get zeros), 32-byte aligned.
 * N % 128 == 0, K % 128 == 0.
 */
int grouped_gemm_mxfp8_dw(const uint8_t *gt_codes, const uint8_t *gt_scales,
                          const uint8_t *xt_codes, const uint8_t *xt_scales,
                          const int32_t *group_offsets, int32_t E,
                          int64_t M_total, int64_t N, int64_t K,
                          float *dw,
                          void *workspace, size_t workspace_bytes, nv_stream_t stream);

/* ---- kernel choice for the three grouped GEMMs (no counterpart in the paper) --
 * 0: automatic (the default): for the MXFP8 GEMMs, CTA pairs with 256 x 256
 *    tiles where the shape allows it (output columns, and for wgrad N,
 *    multiples of 256) and, for dgrad, the experts average at least 512 rows;
 *    otherwise (and for the NVFP4 forward GEMM) two CTAs per SM with
 *    128 x 128 tiles.
 * 1: one CTA per SM, 128 x 128 tiles, two accumulators.
 * 2: two CTAs per SM, 128 x 128 tiles.
 * 3: CTA pairs with 256 x 256 tiles wherever the shape allows it, else 2.
 * 4: CTA pairs with 256 x 128 tiles (two pairs per SM pair) wherever the
 *    shape allows it, else 2.
 * The environment variable NVFP4MOE_GEMM_VARIANT (read at the first GEMM
 * call) gives the initial setting.  Applies to later launches from every host
 * thread; set it while no other thread launches a GEMM.  Returns NV_OK, or
 * NV_ERR_ARG (setting unchanged) for any other value.  Every choice computes
 * the same contraction with fp32 accumulation; summation order differs. */
int nvfp4moe_set_gemm_kernel(int variant);

/* Iteration limit of the grouped GEMMs' pipeline waits (the producer, MMA and
 * epilogue roles waiting on one another's mbarriers), for testing the
 * bounded-wait path: with a limit far below a healthy wait's length the
 * waits run out, the kernel records NV_ERR_TIMEOUT in the status word, every
 * role leaves its loop, and the CTA still waits (with a separate, fixed
 * bound) for the copies and MMAs it has in flight before it frees its tensor
 * memory and exits; the outputs are then incomplete.  spins: 1 .. 2^26, or 0
 * for the default (2^26 polls, far longer than any healthy wait).  Applies to
 * later GEMM launches from every host thread.  Returns NV_OK, or NV_ERR_ARG
 * (setting unchanged) outside that range. */
int nvfp4moe_set_gemm_wait_limit(int64_t spins);

/* ---- Four Over Six: two candidate block scales for activations ------------------------
 * "Recipe details": the activation quantizer selects between two scale
 * factors per block (Four Over Six).  The pages do not state the selection
 * rule; this library takes: each 16-value block is quantized twice under the
 * same outer scale -- block maximum mapped to 6 (nvfp4_quantize's rule,
 * s = RN_E4M3(bamax / fp32(6 sg))) and to 4 (s = RN_E4M3(bamax / fp32(4 sg)),
 * saturating at 448) -- and keeps the candidate with the smaller squared
 * error err = sum_i fp32(x_i - d_i)^2, d_i = fp32(fp32(e2m1_i * s) * sg),
 * summed in fp32 in element order with every operation rounded on its own;
 * ties keep 6.  Same arguments, layouts, outputs and errors as
 * nvfp4_quantize and nvfp4_quantize_requant (the re-quantization reads the
 * codes and scales this rule chose).
 */
int nvfp4_quantize_four_over_six(const void *x, int64_t batch, int64_t rows, int64_t cols,
                                 const int32_t *group_offsets, int32_t num_groups,
                                 const float *outer_scale_in, float *outer_scale_out,
                                 uint8_t *codes, uint8_t *scales,
                                 void *workspace, size_t workspace_bytes, nv_stream_t stream);
int nvfp4_quantize_requant_four_over_six(const void *x, int64_t batch, int64_t rows, int64_t cols,
                                         const int32_t *group_offsets, int32_t num_groups,
                                         const float *outer_scale_in, float *outer_scale_out,
                                         uint8_t *codes, uint8_t *scales,
                                         void *workspace, size_t workspace_bytes,
                                         uint64_t seed, uint64_t counter_offset,
                                         uint8_t *out_codes, uint8_t *out_scales, nv_stream_t stream);

/* ---- per-token activation outer scales ----------------------------------------------
 * "Recipe details": activations get one FP32 outer scale per token (weights
 * one per expert), which keeps a token's quantization independent of the rest
 * of the batch.  Row r of an activation matrix takes
 *   sg_r = amax_r / 2688   (1 for an all-zero row)
 * and is quantized exactly as nvfp4_quantize quantizes a one-row tensor; the
 * dequantized value is fp32(fp32(e2m1 * e4m3) * sg_r).  These calls are the
 * per-token forms of nvfp4_quantize, nvfp4_quantize_requant,
 * dequant_transpose_requant_sr, grouped_gemm_nvfp4_fwd and
 * grouped_gemm_nvfp4_fwd_swiglu (single matrix, no batch), with the same
 * layouts, shape rules and errors as those, except:
 *   sg_rows_in / sg_rows_out: fp32 [rows] device arrays (4-byte aligned).
 *     sg_rows_in NULL -> the per-row amax pass (one extra read of x) writes
 *     sg_rows_out, which must then be non-NULL (else NV_ERR_ARG); sg_rows_in
 *     set -> those scales are used (and copied to sg_rows_out when that is a
 *     different non-NULL array).
 *   The transposed re-quantization forms the per-token dequantized values
 *   first and takes each 32-token block's E8M0 scale from their maximum.
 *   grouped_gemm_nvfp4_fwd_rows: y = acc * fp32(sg_r * sg_w[e]) per row.
 *   grouped_gemm_nvfp4_fwd_swiglu_rows: h_sg_rows fp32 [M_total] receives the
 *     per-token outer scales of h (max |h| of each row, then the rule above;
 *     the array is cleared by the call).
 * Nothing is allocated; every call only enqueues work on `stream`.
 */
int nvfp4_quantize_rows(const void *x, int64_t rows, int64_t cols,
                        const int32_t *group_offsets, int32_t num_groups,
                        const float *sg_rows_in, float *sg_rows_out,
                        uint8_t *codes, uint8_t *scales, nv_stream_t stream);
int nvfp4_quantize_requant_rows(const void *x, int64_t rows, int64_t cols,
                                const int32_t *group_offsets, int32_t num_groups,
                                const float *sg_rows_in, float *sg_rows_out,
                                uint8_t *codes, uint8_t *scales,
                                uint64_t seed, uint64_t counter_offset,
                                uint8_t *out_codes, uint8_t *out_scales, nv_stream_t stream);
int dequant_transpose_requant_sr_rows(const uint8_t *codes, const uint8_t *scales,
                                      const float *sg_rows, int64_t rows, int64_t cols,
                                      const int32_t *group_offsets, int32_t num_groups,
                                      uint64_t seed, uint64_t counter_offset,
                                      uint8_t *out_codes, uint8_t *out_scales, nv_stream_t stream);
int grouped_gemm_nvfp4_fwd_rows(const float *x_sg_rows, const uint8_t *x_codes, const uint8_t *x_scales,
                                const uint8_t *w_codes, const uint8_t *w_scales,
                                const float *w_outer_scale,
                                const int32_t *group_offsets, int32_t E,
                                int64_t M_total, int64_t N, int64_t K,
                                void *y, int y_dtype, nv_stream_t stream);
int grouped_gemm_nvfp4_fwd_swiglu_rows(const float *x_sg_rows, const uint8_t *x_codes,
                                       const uint8_t *x_scales, const uint8_t *w_codes,
                                       const uint8_t *w_scales, const float *w_outer_scale,
                                       const int32_t *group_offsets, int32_t E,
                                       int64_t M_total, int64_t I, int64_t K,
                                       void *y13, void *h, float *h_sg_rows, nv_stream_t stream);

/* ---- 32-point random Hadamard transform + block-scaled S2F6 -------------
 * "Quantized communications": the data of the combine direction is rotated by
 * a 32-dimensional random Hadamard transform and quantized to S2F6 (two signed
 * integer bits, six fractional bits: value k/64, k in [-128, 127]) with one
 * UE8M0 scale per 32 values (8.25 bits per value); the receiver dequantizes
 * and inverts the transform.  The pages state neither the random sign source
 * nor the scale rule; this library takes:
 *   y = H (d * x) / sqrt(32) per block of 32 consecutive values of a row, H
 *       the Sylvester Hadamard matrix, d[i] = -1 where bit i of `signs` is set;
 *       computed in fp32 as the butterfly (a, b) -> (a + b, a - b) over value
 *       bits 0..4 in that order, then one multiply by fp32(1/sqrt(32));
 *   scale e = floor(log2(block max |y|)) clamped to [-127, 127] (code e + 127;
 *       an all-zero block gets code 0), k = RN(y * 2^-e * 64) ties to even,
 *       saturating to [-128, 127];
 *   inverse x = d * (H (k / 64 * 2^e)) / sqrt(32) in the same fp32 order.
 * x bf16 [rows][cols], codes int8 [rows][cols], scales uint8 [rows][cols / 32]
 * (row-major, no swizzle: not an MMA operand), y bf16 or fp32 [rows][cols]
 * (y_dtype NV_OUT_BF16 or NV_OUT_FP32); x, codes and y 32-byte aligned (the
 * kernels move 32 bytes per access); cols % 32 == 0.  All buffers are device
 * memory owned by the caller; the call only enqueues work on `stream` (no
 * allocation, no synchronization).  Returns NV_OK (also for rows or cols 0),
 * NV_ERR_ARG (null pointer, negative size, unknown y_dtype), NV_ERR_SHAPE
 * (cols % 32 != 0), NV_ERR_ALIGN, or NV_ERR_CUDA (launch failure); nothing is
 * written on error.  No counterpart of the kernels themselves on the pages
 * (their conversions are PTX instructions this toolkit does not accept; the
 * rounding is written out).
 */
int rht32_s2f6_quantize(const void *x, int64_t rows, int64_t cols, uint32_t signs,
                        int8_t *codes, uint8_t *scales, nv_stream_t stream);
int s2f6_dequantize_rht32_inverse(const int8_t *codes, const uint8_t *scales,
                                  int64_t rows, int64_t cols, uint32_t signs,
                                  void *y, int y_dtype, nv_stream_t stream);

/* ---- the w2 forward GEMM with RHT-32 + S2F6 in its epilogue ----------------------------
 * "Quantized communications": the combine direction quantizes the experts'
 * output with the 32-point random Hadamard transform and block-scaled S2F6
 * in the down-projection (w2) GEMM's epilogue.  The GEMM of
 * grouped_gemm_nvfp4_fwd with bf16 output (same arguments, layouts and shape
 * rules), and in the same kernel the rht32_s2f6_quantize of every output row
 * (same `signs`): codes and scales bit-identical to the two calls in
 * sequence.
 *   y:      bf16 [M_total][N] (32-byte aligned), or NULL: no bf16 output.
 *   codes:  int8 [M_total][N] (32-byte aligned); scales: u8 [M_total][N / 32].
 * Always runs the 128 x 128 one-SM kernel (whatever nvfp4moe_set_gemm_kernel
 * chose).  Returns as grouped_gemm_nvfp4_fwd; only enqueues work on `stream`.
 */
int grouped_gemm_nvfp4_fwd_rht_s2f6(const float *x_outer_scale, const uint8_t *x_codes,
                                    const uint8_t *x_scales, const uint8_t *w_codes,
                                    const uint8_t *w_scales, const float *w_outer_scale,
                                    const int32_t *group_offsets, int32_t E,
                                    int64_t M_total, int64_t N, int64_t K, uint32_t signs,
                                    void *y, int8_t *codes, uint8_t *scales, nv_stream_t stream);

/* ---- SwiGLU between the expert GEMMs (Figure 5: w13 GEMM, Q, w2 GEMM) -----
 * y13 bf16 [M][2I] (gate columns 0..I-1, up columns I..2I-1);
 * h = bf16(silu(gate) * up) computed in fp32, silu(x) = x / (1 + exp(-x)).
 * Backward: dy13 = [dh * up * silu'(gate), dh * silu(gate)] as bf16.
 * I % 8 == 0. */
int nvfp4moe_swiglu_fwd(const void *y13, int64_t M, int64_t I, void *h, nv_stream_t stream);
int nvfp4moe_swiglu_bwd(const void *dh, const void *y13, int64_t M, int64_t I,
                        void *dy13, nv_stream_t stream);

/* ---- status ------------------------------------------------------------------ */

/* Synchronizes `stream`, returns the first error code any kernel recorded on
 * the current device since the last call (NV_OK if none) and clears it. */
int nvfp4moe_get_device_status(nv_stream_t stream);

/* Self-test of the bounded-wait path: launches one CTA that waits on an
 * mbarrier nothing arrives at, with an iteration limit of `spins`; the wait
 * runs out, the kernel records NV_ERR_TIMEOUT and returns.  No fault, no
 * hang.  1 <= spins <= 2^20 (about a millisecond of polling), else NV_ERR_ARG
 * and nothing is launched, so no caller can keep a CTA spinning for long.
 * Returns the launch status. */
int nvfp4moe_selftest_wait_timeout(int64_t spins, nv_stream_t stream);

/* Diagnostic: the library's stochastic rounding to E4M3 on caller-given
 * values and draws, exactly as the SR kernels apply it ("Re-quantization with
 * stochastic rounding"; the rule and draw convention at the top of this
 * header).  x: fp32 [4 n4] (16-byte aligned); draws: [n4], word i =
 * U_a | U_b << 16, the 16-bit draws of the two pairs (4i, 4i+1) and
 * (4i+2, 4i+3): values 4i and 4i+2 round with U_a and U_b, values 4i+1 and
 * 4i+3 with bitrev16(U_a) and bitrev16(U_b); codes: u8 [4 n4] E4M3
 * (saturating at 448).  Lets a test hold Blackwell's SR conversion to the
 * rule draw by draw. */
int nvfp4moe_sr_e4m3x4(const float *x, const uint32_t *draws, int64_t n4, uint8_t *codes,
                       nv_stream_t stream);

/* Static description of a status code (never NULL). */
const char *nvfp4moe_status_string(int status);

/* Library version string. */
const char *nvfp4moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4MOE_H */
