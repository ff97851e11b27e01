"""Shared plumbing for the GPU parity tests: run a library call on the device
and read its buffers back; run the oracle on the same inputs.  The two sides
share only the seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

from oracle import layout as L
from oracle import nvfp4 as NV
from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N

CANARY = 0xA5


def dev():
    return torch.device("cuda")


def filled(nbytes: int, value: int = CANARY):
    return torch.full((max(int(nbytes), 1),), value, dtype=torch.uint8, device=dev())


def check_status():
    s = N.nvfp4moe_get_device_status()
    assert s == 0, f"device status {s} ({N.status_string(s)})"


def bf16_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().float().numpy()


# ---- NVFP4 quantize ------------------------------------------------------------
def gpu_nvfp4(x: torch.Tensor, batch: int, rows: int, cols: int, groups: torch.Tensor | None = None,
              sg_in: torch.Tensor | None = None):
    E = None if groups is None else groups.numel() - 1
    cb, sb = N.nvfp4_sizes(batch, rows, cols, E)
    codes, scales = filled(cb), filled(sb)
    sg_out = torch.full((batch,), -1.0, dtype=torch.float32, device=dev())
    ws = filled(N.nvfp4moe_quantize_workspace_bytes(batch, rows, cols), 0)
    N.nvfp4_quantize(x, batch, rows, cols, groups, sg_in, sg_out, codes, scales, None if sg_in is not None else ws)
    check_status()
    return codes.cpu().numpy(), scales.cpu().numpy(), sg_out.cpu().numpy()


def oracle_nvfp4(xf: np.ndarray, batch: int, rows: int, cols: int, groups=None, sg_in=None):
    """Expected (packed codes, full scale buffer, sg [batch])."""
    xb = xf.reshape(batch, rows, cols)
    codes, scales, sgs = [], [], []
    for b in range(batch):
        sg = None if sg_in is None else np.float32(sg_in[b])
        c, s, sg = NV.quantize(xb[b], sg)
        codes.append(NV.pack(c))
        scales.append(s)
        sgs.append(sg)
    codes = np.concatenate(codes).reshape(-1)
    logical = np.concatenate(scales)
    if groups is None:
        rmap = L.batched_row_map(batch, rows)
        prow = batch * L.roundup(rows, 128)
    else:
        rmap = L.grouped_row_map(groups)
        prow = L.padded_cap(rows, len(groups) - 1)
    buf = L.swizzle(logical, rmap, prow)
    return codes, buf, np.array(sgs, dtype=np.float32)


def unpack_gpu_nvfp4(codes: np.ndarray, scales: np.ndarray, batch: int, rows: int, cols: int, groups=None):
    """Logical (4-bit codes [batch*rows, cols], scales [batch*rows, cols/16])."""
    c = NV.unpack(codes.reshape(batch * rows, cols // 2))
    rmap = L.batched_row_map(batch, rows) if groups is None else L.grouped_row_map(groups)
    return c, L.unswizzle(scales, rmap, cols // 16)
