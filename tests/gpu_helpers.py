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

# Guard regions: every device buffer a GPU test hands to the library as an
# output (and the layers' own buffers, see conftest) is the front of a larger
# allocation whose last GUARD bytes hold GUARD_BYTE.  A write past the end of
# the buffer changes them; check_guards() (run by check_status() after every
# call and at the end of every GPU test) finds it.  This stands in for a
# memory checker, which is not available here.
GUARD = 4096
GUARD_BYTE = 0xA5
_GUARDED: list = []  # (allocation, bytes in front of the guard)


def dev():
    return torch.device("cuda")


def guarded_bytes(nbytes: int, value=None) -> torch.Tensor:
    """uint8 device buffer of `nbytes` (filled with `value` when given)
    followed by the guard region."""
    n = max(int(nbytes), 1)
    base = torch.empty(n + GUARD, dtype=torch.uint8, device=dev())
    base[n:] = GUARD_BYTE
    if value is not None:
        base[:n] = value
    _GUARDED.append((base, n))
    return base[:n]


def _shape(size):
    return tuple(size) if isinstance(size, (tuple, list, torch.Size)) else (int(size),)


def gempty(size, dtype=torch.float32, device=None):
    """torch.empty with a guard region after the tensor (CUDA only)."""
    if device is not None and torch.device(device).type != "cuda":
        return torch.empty(size, dtype=dtype, device=device)
    shape = _shape(size)
    numel = 1
    for d in shape:
        numel *= int(d)
    nbytes = numel * torch.empty((), dtype=dtype).element_size()
    return guarded_bytes(max(nbytes, 1))[:nbytes].view(dtype).view(shape)


def gfull(size, fill_value, dtype=torch.float32, device=None):
    """torch.full with a guard region after the tensor (CUDA only)."""
    t = gempty(size, dtype=dtype, device=device)
    t.fill_(fill_value)
    return t


def check_guards():
    for base, n in _GUARDED:
        bad = int((base[n:] != GUARD_BYTE).sum())
        assert bad == 0, f"{bad} guard bytes past the end of a {n}-byte output buffer were overwritten"


def clear_guards():
    _GUARDED.clear()


def filled(nbytes: int, value: int = CANARY):
    return guarded_bytes(nbytes, value)


def check_status():
    s = N.nvfp4moe_get_device_status()
    assert s == 0, f"device status {s} ({N.status_string(s)})"
    check_guards()


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
