"""Device buffers and the order of library calls for the hot path.

Every step runs in libnvfp4moe.so; this module only allocates device memory
(through PyTorch) and enqueues the C-ABI calls on the current stream.

SingleLinear   one quantized expert linear layer, forward and backward
               ("End-to-End 4-Bit Training", Figure 4 of the Chinese
               translation): NVFP4 x and w, FPROP NVFP4 GEMM, dequantize ->
               transpose -> SR re-quantize both to MXFP8, SR-quantize the BF16
               gradient row-wise and transposed, DGRAD and WGRAD MXFP8 GEMMs.
MoELayer       the routed experts of one MoE layer (Figure 5: w13 GEMM, Q,
               w2 GEMM) forward and backward on grouped rows: every step of
               the single layer, for the gate/up (w13) and down (w2)
               projections, with SwiGLU between them.
HostStaged     MoELayer steps fed from pinned host memory: the copies in of
               step i+1 and out of step i-1 run on their own streams while
               step i computes (two device slots per staged tensor).
"""
from __future__ import annotations

import torch

from . import nvfp4moe as N

U8 = torch.uint8
BF16 = torch.bfloat16
F32 = torch.float32

# Philox counter offsets of the stochastic roundings of one backward pass
OFF_W13, OFF_W2, OFF_XQ, OFF_HQ, OFF_G2_ROW, OFF_G2_T, OFF_DY13_ROW, OFF_DY13_T = range(8)


def _u8(n, dev):
    return torch.empty(max(int(n), 16), dtype=U8, device=dev)


def _empty(shape, dtype, dev):
    """Every output buffer of the layers comes from here (and _u8)."""
    return torch.empty(shape, dtype=dtype, device=dev)


class NvTensor:
    """NVFP4 codes + block scales + outer scale(s) of a [batch][rows][cols]
    matrix (grouped layout when E is given)."""

    def __init__(self, batch, rows, cols, dev, E=None):
        cb, sb = N.nvfp4_sizes(batch, rows, cols, E)
        self.batch, self.rows, self.cols, self.E = batch, rows, cols, E
        self.codes, self.scales = _u8(cb, dev), _u8(sb, dev)
        self.sg = _empty(batch, F32, dev)
        self.ws = _u8(N.nvfp4moe_quantize_workspace_bytes(batch, rows, cols), dev)
        self.gws = None  # the gathered quantization's workspace, sized on first use

    def gather_workspace(self, src_rows):
        n = N.nvfp4moe_quantize_gather_workspace_bytes(src_rows, self.rows, self.cols)
        if self.gws is None or self.gws.numel() < n:
            self.gws = _u8(n, self.codes.device)
        return self.gws

    def quantize(self, x, groups=None, stream=None, sg_in=None, four_six=False):
        """`sg_in`: a given outer scale (skips the amax pass); `four_six`: the
        Four Over Six block rule."""
        f = N.nvfp4_quantize_four_over_six if four_six else N.nvfp4_quantize
        f(x, self.batch, self.rows, self.cols, groups, sg_in, self.sg, self.codes, self.scales, self.ws, stream)

    def quantize_requant(self, x, mx, seed, offset, groups=None, stream=None, sg_in=None, four_six=False,
                         x_rows=None):
        """quantize() plus the SR re-quantization of the result into `mx`
        (an MxTransposed), in one pass over x.  `x_rows` (int32 [rows]): row
        r of the matrix is x[x_rows[r]] (grouped, per-tensor scale only)."""
        if x_rows is not None:
            if four_six or groups is None:
                raise ValueError("gathered rows: grouped layout and the plain block rule only")
            ws = self.gather_workspace(x.shape[0])
            N.nvfp4_quantize_requant_gather(x, x_rows, x.shape[0], self.rows, self.cols, groups, sg_in, self.sg,
                                            self.codes, self.scales, ws, seed, offset, mx.codes, mx.scales, stream)
            return
        f = N.nvfp4_quantize_requant_four_over_six if four_six else N.nvfp4_quantize_requant
        f(x, self.batch, self.rows, self.cols, groups, sg_in, self.sg, self.codes, self.scales, self.ws, seed, offset,
          mx.codes, mx.scales, stream)


class MxTransposed:
    """MXFP8 transposed operand: [cols][P] grouped (E given) or
    [batch][cols][rows] for weights."""

    def __init__(self, rows, cols, dev, E=None, batch=1):
        if E is not None:
            self.P, cb, sb = N.mxfp8_t_sizes(rows, cols, E)
        else:
            cb, sb = N.requant_weight_sizes(batch, rows, cols)
            self.P = None
        self.codes, self.scales = _u8(cb, dev), _u8(sb, dev)


class MxRows:
    """MXFP8 row-wise operand [rows][cols], grouped scale layout."""

    def __init__(self, rows, cols, dev, E=None):
        cb, sb = N.mxfp8_row_sizes(rows, cols, E)
        self.codes, self.scales = _u8(cb, dev), _u8(sb, dev)


class SingleLinear:
    """y = x_q w_q^T; dx = g w_q; dw = g^T x_q for x [T, d_in], w [d_out, d_in]."""

    def __init__(self, tokens, d_in, d_out, device="cuda"):
        dev = torch.device(device)
        self.T, self.din, self.dout = tokens, d_in, d_out
        self.groups = torch.tensor([0, tokens], dtype=torch.int32, device=dev)
        self.xq = NvTensor(1, tokens, d_in, dev, E=1)
        self.wq = NvTensor(1, d_out, d_in, dev)
        self.y = _empty((tokens, d_out), F32, dev)
        self.xt = MxTransposed(tokens, d_in, dev, E=1)
        self.wt = MxTransposed(d_out, d_in, dev)
        self.g_row = MxRows(tokens, d_out, dev, E=1)
        self.gt = MxTransposed(tokens, d_out, dev, E=1)
        self.dx = _empty((tokens, d_in), F32, dev)
        self.dw = _empty((d_out, d_in), F32, dev)

    def enqueue(self, x, w, g, seed=0, stream=None):
        """x and w are quantized with their SR re-quantizations for the
        backward in the same passes (bit-identical to nvfp4_quantize followed
        by dequant_transpose_requant_sr; two launches fewer for a layer this
        small, whose time is mostly launches)."""
        T, din, dout, go = self.T, self.din, self.dout, self.groups
        self.xq.quantize_requant(x, self.xt, seed, 1, go, stream)
        self.wq.quantize_requant(w, self.wt, seed, 0, None, stream)
        N.grouped_gemm_nvfp4_fwd(None, self.xq.sg, self.xq.codes, self.xq.scales, self.wq.codes, self.wq.scales,
                                 self.wq.sg, go, 1, T, dout, din, self.y, N.NV_OUT_FP32, None, stream)
        N.mxfp8_quantize(g, T, dout, go, N.NV_SR, seed, 2, 3, self.g_row.codes, self.g_row.scales,
                         self.gt.codes, self.gt.scales, stream)
        N.grouped_gemm_mxfp8_dx(self.g_row.codes, self.g_row.scales, self.wt.codes, self.wt.scales, go, 1, T, dout,
                                din, self.dx, N.NV_OUT_FP32, None, stream)
        N.grouped_gemm_mxfp8_dw(self.gt.codes, self.gt.scales, self.xt.codes, self.xt.scales, go, 1, T, dout, din,
                                self.dw, None, stream)

    def run(self, x, w, g, seed=0):
        """Enqueue the layer and return its outputs on the host (numpy)."""
        self.enqueue(x, w, g, seed)
        torch.cuda.synchronize()
        T, din, dout = self.T, self.din, self.dout
        P = self.xt.P
        return {
            "x_sg": self.xq.sg.cpu().numpy()[0], "w_sg": self.wq.sg.cpu().numpy()[0],
            "x_codes": self.xq.codes[: T * din // 2].cpu().numpy().reshape(T, din // 2),
            "w_codes": self.wq.codes[: dout * din // 2].cpu().numpy().reshape(dout, din // 2),
            "y": self.y.cpu().numpy(),
            "wt_codes": self.wt.codes[: din * dout].cpu().numpy(),
            "g_codes": self.g_row.codes[: T * dout].cpu().numpy(),
            "P": P,
            "gt_codes": self.gt.codes[: dout * P].cpu().numpy(), "gt_scales": self.gt.scales.cpu().numpy(),
            "xt_codes": self.xt.codes[: din * P].cpu().numpy(), "xt_scales": self.xt.scales.cpu().numpy(),
            "dx": self.dx.cpu().numpy(), "dw": self.dw.cpu().numpy(),
        }


class MoELayer:
    """Routed experts of one MoE layer: rows grouped by expert (group_offsets),
    w13 [E][2I][d] (gate rows then up rows), w2 [E][d][I].

    A training step (`step`) quantizes each forward tensor with
    nvfp4_quantize_requant, so the MXFP8 re-quantized operands of the
    backward come out of the forward's quantization pass; `fuse_requant=False`
    runs nvfp4_quantize in the forward and the four
    dequant_transpose_requant_sr calls in the backward instead.  The w13 GEMM
    computes SwiGLU and the outer scale of h in its epilogue
    (grouped_gemm_nvfp4_fwd_swiglu) when d_ff % 128 == 0; `fuse_swiglu=False`
    runs the GEMM, nvfp4moe_swiglu_fwd and the amax pass of h instead.  The
    dgrad of w2 applies the SwiGLU backward in its epilogue
    (grouped_gemm_mxfp8_dx_swiglu_bwd, dh never stored) when d_ff % 128 == 0;
    `fuse_swiglu_bwd=False` stores dh and runs nvfp4moe_swiglu_bwd.  Every
    choice gives the same results, bit for bit.

    `per_token=True` quantizes the activations x and h with one outer scale
    per token (the *_rows calls; weights keep one per expert), the recipe's
    batch-invariant form; `four_over_six=True` quantizes them with the Four
    Over Six block rule.  Both change the results."""

    def __init__(self, M, d_model, d_ff, E, device="cuda", backward=True, fuse_requant=True, fuse_swiglu=True,
                 per_token=False, four_over_six=False, overlap_amax=False, fuse_swiglu_bwd=True):
        if per_token and four_over_six:
            raise ValueError("per-token scales and Four Over Six are separate options")
        dev = torch.device(device)
        self.M, self.d, self.I, self.E = M, d_model, d_ff, E
        I2 = 2 * d_ff
        # forward
        self.xq = NvTensor(1, M, d_model, dev, E=E)
        self.w13q = NvTensor(E, I2, d_model, dev)
        self.w2q = NvTensor(E, d_model, d_ff, dev)
        self.y13 = _empty((M, I2), BF16, dev)
        self.h = _empty((M, d_ff), BF16, dev)
        self.hq = NvTensor(1, M, d_ff, dev, E=E)
        self.y2 = _empty((M, d_model), BF16, dev)
        self.fuse_swiglu = fuse_swiglu and d_ff % 128 == 0
        self.h_sg = _empty(1, F32, dev)  # outer scale of h from the fused epilogue
        self.per_token = per_token
        self.four_six = four_over_six
        # overlap_amax: the per-tensor amax passes of w13, w2 and x (HBM-bound)
        # run on a side stream, each overlapping the quantization (ALU-bound)
        # of the tensor before it, and the quantizers take the scales as given
        # (same results; measured no faster at the MoE shapes: 9.11 against
        # 9.05 ms per step, so off by default)
        self.side = torch.cuda.Stream(dev) if overlap_amax and not per_token else None
        if per_token:
            self.x_sg_rows = _empty(M, F32, dev)
            self.h_sg_rows = _empty(M, F32, dev)
        self.fuse_requant = fuse_requant and backward
        self.fuse_swiglu_bwd = fuse_swiglu_bwd and d_ff % 128 == 0
        self._requant_seed = None  # seed of the operands the last forward re-quantized
        if not backward:  # forward-only use (sampling): no backward buffers
            return
        # backward
        self.xt = MxTransposed(M, d_model, dev, E=E)
        self.ht = MxTransposed(M, d_ff, dev, E=E)
        self.w13t = MxTransposed(I2, d_model, dev, batch=E)
        self.w2t = MxTransposed(d_model, d_ff, dev, batch=E)
        self.g2_row = MxRows(M, d_model, dev, E=E)
        self.g2t = MxTransposed(M, d_model, dev, E=E)
        self.dh = None if self.fuse_swiglu_bwd else _empty((M, d_ff), BF16, dev)
        self.dy13 = _empty((M, I2), BF16, dev)
        self.dy13_row = MxRows(M, I2, dev, E=E)
        self.dy13t = MxTransposed(M, I2, dev, E=E)
        self.dx = _empty((M, d_model), BF16, dev)
        self.dw2 = _empty((E, d_model, d_ff), F32, dev)
        self.dw13 = _empty((E, I2, d_model), F32, dev)

    @property
    def gathers_rows(self):
        """Whether step() can take the tokens and the routed rows' source map
        (the quantization of x gathering the rows): the fused training step
        with per-tensor scales, the plain block rule and no side stream."""
        return self.fuse_requant and not self.per_token and not self.four_six and self.side is None

    # GEMM FLOPs of one forward (2 GEMMs) and one backward (4 GEMMs)
    def flops(self):
        fwd = 2 * self.M * (2 * self.I) * self.d + 2 * self.M * self.d * self.I
        return fwd, 2 * fwd

    def quantize_weights(self, w13, w2, stream=None, seed=None):
        """NVFP4 of both expert weight stacks, one outer scale per expert
        (plus their MXFP8 re-quantization when `seed` is given)."""
        if seed is None:
            self.w13q.quantize(w13, None, stream)
            self.w2q.quantize(w2, None, stream)
        else:
            self.w13q.quantize_requant(w13, self.w13t, seed, OFF_W13, None, stream)
            self.w2q.quantize_requant(w2, self.w2t, seed, OFF_W2, None, stream)

    def forward(self, x, w13, w2, groups, stream=None, seed=None, x_rows=None):
        """`seed` (training): also re-quantize the forward tensors for the
        backward in the same passes.  `x_rows` (int32 [M]): x holds the
        tokens and routed row r is token x_rows[r] (the dispatch), gathered
        by the quantization of x itself (training step, per-tensor scales)."""
        seed = seed if self.fuse_requant else None
        if x_rows is not None and (seed is None or not self.gathers_rows):
            raise ValueError("gathered activations need the fused training step with per-tensor scales")
        x_sg = None
        if self.side is not None:
            main = stream if stream is not None else torch.cuda.current_stream()
            start = torch.cuda.Event()
            start.record(main)
            self.side.wait_event(start)
            ready = []
            for t, q in ((w13, self.w13q), (w2, self.w2q), (x, self.xq)):
                N.nvfp4_outer_scale(t, q.batch, q.rows * q.cols, q.sg, q.ws, self.side)
                ev = torch.cuda.Event()
                ev.record(self.side)
                ready.append(ev)
            for ev, (t, q, mx, off) in zip(ready[:2], ((w13, self.w13q, getattr(self, "w13t", None), OFF_W13),
                                                       (w2, self.w2q, getattr(self, "w2t", None), OFF_W2))):
                main.wait_event(ev)
                if seed is None:
                    q.quantize(t, None, stream, sg_in=q.sg)
                else:
                    q.quantize_requant(t, mx, seed, off, None, stream, sg_in=q.sg)
            main.wait_event(ready[2])
            x_sg = self.xq.sg
        else:
            self.quantize_weights(w13, w2, stream, seed)
        self.forward_activations(x, groups, stream, seed, x_sg=x_sg, x_rows=x_rows)
        self._requant_seed = seed

    def forward_activations(self, x, groups, stream=None, seed=None, x_sg=None, x_rows=None):
        """The forward with the weights already quantized (e.g. sampling);
        `x_sg`: x's outer scale, already computed; `x_rows`: see forward."""
        if self.per_token:
            return self._forward_activations_rows(x, groups, stream, seed)
        M, d, I, E = self.M, self.d, self.I, self.E
        f6 = self.four_six
        if seed is None:
            self.xq.quantize(x, groups, stream, sg_in=x_sg, four_six=f6)
        else:
            self.xq.quantize_requant(x, self.xt, seed, OFF_XQ, groups, stream, sg_in=x_sg, four_six=f6,
                                     x_rows=x_rows)
        sg_h = None
        if self.fuse_swiglu:
            N.grouped_gemm_nvfp4_fwd_swiglu(self.xq.sg, self.xq.codes, self.xq.scales, self.w13q.codes,
                                            self.w13q.scales, self.w13q.sg, groups, E, M, I, d, self.y13, self.h,
                                            self.h_sg, stream)
            sg_h = self.h_sg
        else:
            N.grouped_gemm_nvfp4_fwd(None, self.xq.sg, self.xq.codes, self.xq.scales, self.w13q.codes,
                                     self.w13q.scales, self.w13q.sg, groups, E, M, 2 * I, d, self.y13, N.NV_OUT_BF16,
                                     None, stream)
            N.nvfp4moe_swiglu_fwd(self.y13, M, I, self.h, stream)
        if seed is None:
            self.hq.quantize(self.h, groups, stream, sg_in=sg_h, four_six=f6)
        else:
            self.hq.quantize_requant(self.h, self.ht, seed, OFF_HQ, groups, stream, sg_in=sg_h, four_six=f6)
        N.grouped_gemm_nvfp4_fwd(None, self.hq.sg, self.hq.codes, self.hq.scales, self.w2q.codes, self.w2q.scales,
                                 self.w2q.sg, groups, E, M, d, I, self.y2, N.NV_OUT_BF16, None, stream)

    def _forward_activations_rows(self, x, groups, stream, seed):
        M, d, I, E = self.M, self.d, self.I, self.E
        xq, hq, xs, hs = self.xq, self.hq, self.x_sg_rows, self.h_sg_rows
        if seed is None:
            N.nvfp4_quantize_rows(x, M, d, groups, None, xs, xq.codes, xq.scales, stream)
        else:
            N.nvfp4_quantize_requant_rows(x, M, d, groups, None, xs, xq.codes, xq.scales, seed, OFF_XQ,
                                          self.xt.codes, self.xt.scales, stream)
        h_in = None
        if self.fuse_swiglu:
            N.grouped_gemm_nvfp4_fwd_swiglu_rows(xs, xq.codes, xq.scales, self.w13q.codes, self.w13q.scales,
                                                 self.w13q.sg, groups, E, M, I, d, self.y13, self.h, hs, stream)
            h_in = hs
        else:
            N.grouped_gemm_nvfp4_fwd_rows(xs, xq.codes, xq.scales, self.w13q.codes, self.w13q.scales, self.w13q.sg,
                                          groups, E, M, 2 * I, d, self.y13, N.NV_OUT_BF16, stream)
            N.nvfp4moe_swiglu_fwd(self.y13, M, I, self.h, stream)
        if seed is None:
            N.nvfp4_quantize_rows(self.h, M, I, groups, h_in, hs, hq.codes, hq.scales, stream)
        else:
            N.nvfp4_quantize_requant_rows(self.h, M, I, groups, h_in, hs, hq.codes, hq.scales, seed, OFF_HQ,
                                          self.ht.codes, self.ht.scales, stream)
        N.grouped_gemm_nvfp4_fwd_rows(hs, hq.codes, hq.scales, self.w2q.codes, self.w2q.scales, self.w2q.sg, groups,
                                      E, M, d, I, self.y2, N.NV_OUT_BF16, stream)

    def backward(self, g2, groups, seed=3, stream=None, dx_out=None):
        """dx goes to `dx_out` when given (bf16 [M][d_model]), else self.dx."""
        M, d, I, E = self.M, self.d, self.I, self.E
        dx = self.dx if dx_out is None else dx_out
        # re-quantize the saved forward tensors (dequantize -> transpose -> SR to
        # MXFP8), unless the forward already did with this seed
        if self._requant_seed != seed:
            self.requant_saved(groups, seed, stream)
        self._backward_gemms(g2, groups, seed, stream, dx)

    def requant_saved(self, groups, seed, stream=None):
        M, d, I, E = self.M, self.d, self.I, self.E
        I2 = 2 * I
        N.dequant_transpose_requant_sr(self.w13q.codes, self.w13q.scales, self.w13q.sg, E, I2, d, None, seed,
                                       OFF_W13, self.w13t.codes, self.w13t.scales, stream)
        N.dequant_transpose_requant_sr(self.w2q.codes, self.w2q.scales, self.w2q.sg, E, d, I, None, seed, OFF_W2,
                                       self.w2t.codes, self.w2t.scales, stream)
        if self.per_token:
            N.dequant_transpose_requant_sr_rows(self.xq.codes, self.xq.scales, self.x_sg_rows, M, d, groups, seed,
                                                OFF_XQ, self.xt.codes, self.xt.scales, stream)
            N.dequant_transpose_requant_sr_rows(self.hq.codes, self.hq.scales, self.h_sg_rows, M, I, groups, seed,
                                                OFF_HQ, self.ht.codes, self.ht.scales, stream)
            return
        N.dequant_transpose_requant_sr(self.xq.codes, self.xq.scales, self.xq.sg, 1, M, d, groups, seed, OFF_XQ,
                                       self.xt.codes, self.xt.scales, stream)
        N.dequant_transpose_requant_sr(self.hq.codes, self.hq.scales, self.hq.sg, 1, M, I, groups, seed, OFF_HQ,
                                       self.ht.codes, self.ht.scales, stream)

    def _backward_gemms(self, g2, groups, seed, stream, dx):
        M, d, I, E = self.M, self.d, self.I, self.E
        I2 = 2 * I
        # down projection: dh = g2 w2, dW2 = g2^T h_q
        N.mxfp8_quantize(g2, M, d, groups, N.NV_SR, seed, OFF_G2_ROW, OFF_G2_T, self.g2_row.codes,
                         self.g2_row.scales, self.g2t.codes, self.g2t.scales, stream)
        # (fused: the SwiGLU backward in the dgrad's epilogue, dh never stored)
        if self.fuse_swiglu_bwd:
            N.grouped_gemm_mxfp8_dx_swiglu_bwd(self.g2_row.codes, self.g2_row.scales, self.w2t.codes,
                                               self.w2t.scales, groups, E, M, d, I, self.y13, self.dy13, stream)
        else:
            N.grouped_gemm_mxfp8_dx(self.g2_row.codes, self.g2_row.scales, self.w2t.codes, self.w2t.scales, groups,
                                    E, M, d, I, self.dh, N.NV_OUT_BF16, None, stream)
        N.grouped_gemm_mxfp8_dw(self.g2t.codes, self.g2t.scales, self.ht.codes, self.ht.scales, groups, E, M, d, I,
                                self.dw2, None, stream)
        # SwiGLU backward (unless fused above), then gate/up: dx = dy13 w13, dW13 = dy13^T x_q
        if not self.fuse_swiglu_bwd:
            N.nvfp4moe_swiglu_bwd(self.dh, self.y13, M, I, self.dy13, stream)
        N.mxfp8_quantize(self.dy13, M, I2, groups, N.NV_SR, seed, OFF_DY13_ROW, OFF_DY13_T, self.dy13_row.codes,
                         self.dy13_row.scales, self.dy13t.codes, self.dy13t.scales, stream)
        N.grouped_gemm_mxfp8_dx(self.dy13_row.codes, self.dy13_row.scales, self.w13t.codes, self.w13t.scales,
                                groups, E, M, I2, d, dx, N.NV_OUT_BF16, None, stream)
        N.grouped_gemm_mxfp8_dw(self.dy13t.codes, self.dy13t.scales, self.xt.codes, self.xt.scales, groups, E, M,
                                I2, d, self.dw13, None, stream)

    def step(self, x, w13, w2, g2, groups, seed=3, stream=None, dx_out=None, x_rows=None):
        self.forward(x, w13, w2, groups, stream, seed, x_rows=x_rows)
        self.backward(g2, groups, seed, stream, dx_out)

    @staticmethod
    def capture(fn):
        """Capture `fn()` -- this layer's calls on the current stream, e.g.
        `lambda: layer.forward_activations(x, groups)` -- into a CUDA graph
        and return it; `graph.replay()` reruns the same launches on the same
        buffers.  One eager call first sets up what the library does once
        (kernel attributes, occupancy queries, the device status word), none
        of which may run during a capture."""
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g

    def launches_per_step(self, gathered=False, tokens=None):
        """Kernels one step launches: forward = 4 NVFP4 quantizations x 3
        kernels (amax, finalize, quantize or quantize + requant) + 2 GEMMs +
        SwiGLU, or with the SwiGLU epilogue: 3 x 3 + the fused GEMM, the
        outer-scale kernel and one kernel for h + the w2 GEMM; backward = (4
        requants unless fused) + 2 MXFP8 quantizations + 4 GEMMs + SwiGLU
        backward.  `gathered`: x given as tokens + row map; with no more tokens
        than routed rows its amax pass adds the tokens' row-maximum kernel and
        its quantization the tokens' NVFP4 pass (then the routed rows'
        copy + re-quantization)."""
        fwd = (3 * 3 + 2 + 1 + 1) if self.fuse_swiglu else (4 * 3 + 2 + 1)
        if gathered and (tokens is None or tokens <= self.M):
            fwd += 2
        # (with the side-stream amax passes the same kernels run, the amax ones on the side stream)
        if self.per_token:  # x: row amax + quantize; h: from the epilogue's row scales (1) or row amax + quantize
            fwd = (2 + 2 * 3 + 2 + 1 + 1) if self.fuse_swiglu else (2 + 2 * 3 + 2 + 2 + 1)
        # backward: 2 MXFP8 quantizations + 4 GEMMs (+ the SwiGLU backward unless in the dgrad epilogue)
        return fwd + (0 if self.fuse_requant else 4) + (2 + 4 + (0 if self.fuse_swiglu_bwd else 1))


class HostStaged:
    """MoELayer steps whose activations x and upstream gradient g2 come from
    pinned host memory and whose dx goes back to pinned host memory.

    Step i copies its inputs into device slot i % 2 on the copy-in stream (x,
    then g2), computes on the caller's current stream and copies dx out of
    slot i % 2 on the copy-out stream, so the transfers of neighbouring steps
    overlap the compute of step i.  The forward waits only for x and the
    backward for g2, so the g2 copy overlaps the step's own forward.  Events
    order every reuse of a slot: a copy into a slot waits until the step that
    last read that tensor has finished with it (x: its forward, g2: its
    backward), and a backward waits until the copy out of its dx slot (from two
    steps earlier) has finished.
    The host buffers must stay untouched until `synchronize()` (or until the
    copy-out of that step has completed)."""

    def __init__(self, layer: MoELayer, device="cuda", tokens=None):
        """`tokens`: the steps take the token matrix [tokens, d] and the routed
        rows' source tokens (int32 [M]) instead of the routed rows themselves."""
        dev = torch.device(device)
        M, d = layer.M, layer.d
        self.layer = layer
        self.tokens = tokens
        self.x = [torch.empty((tokens if tokens is not None else M, d), dtype=BF16, device=dev) for _ in range(2)]
        self.rows = [torch.empty(M, dtype=torch.int32, device=dev) for _ in range(2)] if tokens is not None else None
        self.g2 = [torch.empty((M, d), dtype=BF16, device=dev) for _ in range(2)]
        self.dx = [_empty((M, d), BF16, dev) for _ in range(2)]
        self.s_in = torch.cuda.Stream(dev)
        self.s_out = torch.cuda.Stream(dev)
        self.x_read = [None, None]      # forward of the slot's last step finished (x free)
        self.g2_read = [None, None]     # backward of the slot's last step finished (g2 free)
        self.out_done = [None, None]    # copy-out of the slot's last dx finished
        self.n = 0

    def bytes_per_step(self):
        """(host -> device, device -> host) bytes of one step."""
        b = lambda t: t.numel() * t.element_size()
        rows = b(self.rows[0]) if self.rows is not None else 0
        return b(self.x[0]) + rows + b(self.g2[0]), b(self.dx[0])

    def step(self, x_h, g2_h, dx_h, w13, w2, groups, seed=3, rows_h=None):
        k = self.n % 2
        comp = torch.cuda.current_stream()
        x_in, g2_in = torch.cuda.Event(), torch.cuda.Event()
        with torch.cuda.stream(self.s_in):
            if self.x_read[k] is not None:
                self.s_in.wait_event(self.x_read[k])
            self.x[k].copy_(x_h, non_blocking=True)
            if self.rows is not None:
                self.rows[k].copy_(rows_h, non_blocking=True)
            x_in.record(self.s_in)
            if self.g2_read[k] is not None:
                self.s_in.wait_event(self.g2_read[k])
            self.g2[k].copy_(g2_h, non_blocking=True)
            g2_in.record(self.s_in)
        comp.wait_event(x_in)
        self.layer.forward(self.x[k], w13, w2, groups, comp, seed,
                           x_rows=self.rows[k] if self.rows is not None else None)
        fwd_done = torch.cuda.Event()
        fwd_done.record(comp)
        self.x_read[k] = fwd_done
        comp.wait_event(g2_in)
        if self.out_done[k] is not None:
            comp.wait_event(self.out_done[k])
        self.layer.backward(self.g2[k], groups, seed, comp, dx_out=self.dx[k])
        done = torch.cuda.Event()
        done.record(comp)
        self.g2_read[k] = done
        self.s_out.wait_event(done)
        with torch.cuda.stream(self.s_out):
            dx_h.copy_(self.dx[k], non_blocking=True)
        out = torch.cuda.Event()
        out.record(self.s_out)
        self.out_done[k] = out
        self.n += 1
        return out

    def synchronize(self):
        for e in self.out_done:
            if e is not None:
                e.synchronize()
