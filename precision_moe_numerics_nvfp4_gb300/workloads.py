"""Seeded synthetic inputs for the expert hot path.

This module only draws random tensors and routes tokens; it holds none of the
quantization or GEMM arithmetic, so both the CUDA path and the CPU oracle can
be fed from it.  Every generator takes a ``torch.Generator``-compatible seed
and a device; the same seed on the same device always gives the same bytes.

Workloads (shapes and distributions of the pages' setting -- a GB300 MoE
layer with 1x16 NVFP4 forward and MXFP8 backward -- made synthetic):
  single_linear      x [256x512] ~N(0,1) with 4 rows x64, w [1024x512]
                     ~N(0,0.02) with 8 elements x100, g [256x1024] ~N(0,1e-3)
  quant_sweep        [8192x8192] and [16384x7168], Student-t(3) x 0.05 with
                     0.01% of elements x1000
  moe_forward        16384 tokens, d_model 4096, 64 experts, top-8 routing
                     from logits ~N(0,1) + bias ~N(0,1); SwiGLU experts
                     gate/up [4096->1536 x2], down [1536->4096], ~N(0,0.02)
  moe_backward       same shapes, down-output gradient ~N(0,1e-3)
  decode             128 experts [7168 x 2048 gate/up/down], 256 tokens plain
                     top-8 (no bias)
The second parameter of N(mean, s) is the standard deviation.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float, gen: torch.Generator, device, dtype=torch.bfloat16):
    return (torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std).to(dtype)


def student_t(shape, nu: int, scale: float, gen: torch.Generator, device):
    """Student-t with integer nu: Z / sqrt(sum_{i<nu} Z_i^2 / nu), times scale."""
    z = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    v = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(nu):
        zi = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        v += zi * zi
    return z / torch.sqrt(v / nu) * scale


def plant_rows(x: torch.Tensor, count: int, factor: float, gen: torch.Generator):
    """Multiply ``count`` distinct random rows by ``factor`` (in place)."""
    idx = torch.randperm(x.shape[0], generator=gen, device=x.device)[:count]
    x[idx] = (x[idx].float() * factor).to(x.dtype)
    return x


def plant_elements(x: torch.Tensor, count: int, factor: float, gen: torch.Generator):
    """Multiply ``count`` distinct random elements by ``factor`` (in place)."""
    flat = x.view(-1)
    idx = torch.randperm(flat.numel(), generator=gen, device=x.device)[:count]
    flat[idx] = (flat[idx].float() * factor).to(x.dtype)
    return x


def route_topk(logits: torch.Tensor, bias: torch.Tensor, k: int):
    """Top-k routing by (logit + bias); ties go to the lower expert id.
    Returns (token of every routed row, sorted by expert then token;
    group_offsets int32 [E+1])."""
    T, E = logits.shape
    score = logits.float() + bias.float()[None, :]
    order = torch.sort(score, dim=1, descending=True, stable=True).indices[:, :k]
    expert = order.reshape(-1)
    token = torch.arange(T, device=logits.device).repeat_interleave(k)
    key = expert.to(torch.int64) * T + token
    perm = torch.argsort(key)
    counts = torch.bincount(expert, minlength=E)
    offsets = torch.zeros(E + 1, dtype=torch.int64, device=logits.device)
    offsets[1:] = torch.cumsum(counts, 0)
    return token[perm], offsets.to(torch.int32)


@dataclass
class SingleLinear:
    x: torch.Tensor   # bf16 [256, 512]
    w: torch.Tensor   # bf16 [1024, 512]
    g: torch.Tensor   # bf16 [256, 1024]


def single_linear(device="cpu", seed: int = 0, tokens: int = 256, d_in: int = 512, d_out: int = 1024):
    gen = _gen(seed, device)
    x = normal((tokens, d_in), 1.0, gen, device)
    plant_rows(x, 4, 64.0, gen)
    w = normal((d_out, d_in), 0.02, gen, device)
    plant_elements(w, 8, 100.0, gen)
    g = normal((tokens, d_out), 1e-3, gen, device)
    return SingleLinear(x, w, g)


def quant_sweep(shape, device="cpu", seed: int = 1, nu: int = 3, scale: float = 0.05,
                outlier_frac: float = 1e-4, outlier_factor: float = 1000.0):
    """One tensor of the quantization sweep (bf16)."""
    gen = _gen(seed, device)
    x = student_t(shape, nu, scale, gen, device)
    n_out = int(np.floor(outlier_frac * x.numel()))
    plant_elements(x, n_out, outlier_factor, gen)
    return x.to(torch.bfloat16)


QUANT_SWEEP_SHAPES = ((8192, 8192), (16384, 7168))


@dataclass
class MoE:
    x_perm: torch.Tensor          # bf16 [T*k, d_model], rows grouped by expert
    group_offsets: torch.Tensor   # int32 [E+1]
    token: torch.Tensor           # int64 [T*k] source token of each row
    w13: torch.Tensor             # bf16 [E, 2I, d_model] (gate rows then up rows)
    w2: torch.Tensor              # bf16 [E, d_model, I]
    g2: torch.Tensor | None       # bf16 [T*k, d_model] gradient of the down output
    x: torch.Tensor | None = None     # bf16 [T, d_model] the tokens (x_perm = x[token])
    rows: torch.Tensor | None = None  # int32 [T*k] source token of each row


def moe(device="cpu", seed: int = 2, tokens: int = 16384, d_model: int = 4096, experts: int = 64,
        topk: int = 8, d_ff: int = 1536, with_grad: bool = False, grad_seed: int = 3,
        weights: bool = True, bias_std: float = 1.0):
    """Routed expert inputs: top-k of logits ~ N(0,1) plus a per-expert bias
    ~ N(0, bias_std) (uneven groups; bias_std 0 gives plain top-k)."""
    gen = _gen(seed, device)
    logits = torch.randn((tokens, experts), generator=gen, device=device)
    bias = torch.randn((experts,), generator=gen, device=device) * bias_std
    token, offsets = route_topk(logits, bias, topk)
    x = normal((tokens, d_model), 1.0, gen, device)
    x_perm = x[token].contiguous()
    w13 = w2 = None
    if weights:
        w_gate = normal((experts, d_ff, d_model), 0.02, gen, device)
        w_up = normal((experts, d_ff, d_model), 0.02, gen, device)
        w13 = torch.cat([w_gate, w_up], dim=1).contiguous()
        del w_gate, w_up
        w2 = normal((experts, d_model, d_ff), 0.02, gen, device)
    g2 = None
    if with_grad:
        gg = _gen(grad_seed, device)
        g2 = normal((tokens * topk, d_model), 1e-3, gg, device)
    return MoE(x_perm, offsets, token, w13, w2, g2, x, token.to(torch.int32))


def decode(device="cpu", seed: int = 4, tokens: int = 256, d_model: int = 7168, d_ff: int = 2048,
           experts: int = 128, topk: int = 8):
    """Sampler-style decode: plain top-8 routing of logits ~ N(0,1), ~16 rows
    per expert (asserted 1..64)."""
    m = moe(device, seed, tokens, d_model, experts, topk, d_ff, bias_std=0.0)
    sizes = torch.diff(m.group_offsets.to(torch.int64))
    if int(sizes.min()) < 1 or int(sizes.max()) > 64:
        raise RuntimeError("decode routing left an expert outside 1..64 rows")
    return m


def fig2_tile(seed: int = 7) -> np.ndarray:
    """A 16x16 tile with one full row of large values: row 0 = sixteen 64.0,
    the other 240 values log-uniform in [0.5, 2.5], 19 of them replaced by
    U[3, 4] (the structure the page's Figure 2 describes; its values are not
    printed)."""
    rng = np.random.default_rng(seed)
    t = np.exp(rng.uniform(np.log(0.5), np.log(2.5), size=(16, 16)))
    t[0, :] = 64.0
    pos = rng.choice(240, size=19, replace=False) + 16
    t.reshape(-1)[pos] = rng.uniform(3.0, 4.0, size=19)
    return t.astype(np.float32)


def fig3_tile(seed: int = 8) -> np.ndarray:
    """A 16x16 tile of log-uniform [0.5, 2.5] values with one 64.0 in the
    last row (the structure of the page's Figure 3)."""
    rng = np.random.default_rng(seed)
    t = np.exp(rng.uniform(np.log(0.5), np.log(2.5), size=(16, 16)))
    t[15, rng.integers(0, 16)] = 64.0
    return t.astype(np.float32)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 patterns of a bf16 tensor (on the host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f32_numpy(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().float().numpy()
