"""Scale-factor memory layout and grouped-row padding.  Test infrastructure
only.

The pages do not fix a layout.  The library stores every block-scale matrix in
the layout that block-scaled tensor-core MMA reads (the "128x4" scale-factor
tile of the PTX ISA's tcgen05 block-scaling section and of cuBLASLt's
block-scaled matmul): logical scale [row r, block column c] of a matrix with
KB block columns lives at

    atom(r // 128, c // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4,
    atom(t, j) = t * ceil(KB / 4) + j

with zero bytes in every padding position.  Rows are first mapped to padded
rows:
  * plain / batched matrices [B][R][...]:  r' = b * roundup(R, 128) + r
  * grouped rows (experts' tokens)      :  r' = P_e + (r - o_e), with o_e the
    group start and P_e = sum_{e' < e} roundup(M_e', 128) ("group-padded")
so that every 128-row tile of a group has its own atoms.  A grouped buffer is
sized for the worst case P_cap = roundup(M_total + 127 E, 128) rows.
"""
from __future__ import annotations

import numpy as np


def roundup(a: int, b: int) -> int:
    return (a + b - 1) // b * b


def padded_cap(M_total: int, E: int) -> int:
    """Rows (or transposed columns) reserved for a grouped layout."""
    return roundup(M_total + 127 * E, 128)


def group_padded_starts(group_offsets):
    """P_e for every group (and the padded total as the last entry)."""
    o = np.asarray(group_offsets, dtype=np.int64)
    sizes = np.diff(o)
    padded = (sizes + 127) // 128 * 128
    return np.concatenate([[0], np.cumsum(padded)]).astype(np.int64)


def atom_offset(rp, c, kblocks: int):
    """Byte offset of the scale of padded row rp, block column c."""
    rp = np.asarray(rp, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    ka = (kblocks + 3) // 4
    return ((rp // 128) * ka + c // 4) * 512 + (rp % 32) * 16 + ((rp // 32) % 4) * 4 + c % 4


def scale_buffer_bytes(padded_rows: int, kblocks: int) -> int:
    return roundup(padded_rows, 128) // 128 * ((kblocks + 3) // 4) * 512


def swizzle(scales, padded_rows_of, total_padded_rows: int) -> np.ndarray:
    """Place a logical scale matrix [R, KB] into a zero-filled buffer.
    ``padded_rows_of`` maps each logical row index to its padded row."""
    s = np.asarray(scales, dtype=np.uint8)
    R, KB = s.shape
    buf = np.zeros(scale_buffer_bytes(total_padded_rows, KB), dtype=np.uint8)
    rp = np.asarray(padded_rows_of, dtype=np.int64)
    rr, cc = np.meshgrid(rp, np.arange(KB), indexing="ij")
    buf[atom_offset(rr, cc, KB)] = s
    return buf


def unswizzle(buf, padded_rows_of, kblocks: int) -> np.ndarray:
    """Read a logical [R, KB] scale matrix out of a swizzled buffer."""
    b = np.asarray(buf, dtype=np.uint8)
    rp = np.asarray(padded_rows_of, dtype=np.int64)
    rr, cc = np.meshgrid(rp, np.arange(kblocks), indexing="ij")
    return b[atom_offset(rr, cc, kblocks)]


def grouped_row_map(group_offsets) -> np.ndarray:
    """Padded row of every logical row of a grouped matrix."""
    o = np.asarray(group_offsets, dtype=np.int64)
    P = group_padded_starts(o)
    out = np.empty(int(o[-1]), dtype=np.int64)
    for e in range(len(o) - 1):
        out[o[e]:o[e + 1]] = P[e] + np.arange(o[e + 1] - o[e])
    return out


def batched_row_map(batch: int, rows: int) -> np.ndarray:
    """Padded row of every row of a [batch][rows] stack of matrices."""
    b = np.arange(batch, dtype=np.int64)[:, None]
    return (b * roundup(rows, 128) + np.arange(rows, dtype=np.int64)[None, :]).reshape(-1)
