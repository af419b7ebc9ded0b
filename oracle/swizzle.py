"""128x4 tiled layout of e8m0 scale factors (CPU oracle).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this file.

The pages say the scale factors are rearranged from a plain row-major matrix
into 128x4 tiles for Blackwell's fifth-generation tensor cores (tcgen05), by a
dedicated kernel ("Accelerating Llama4 Scout training with TorchAO MXFP8 MoE
primitives", section details, and the caption of its 128x4 tile layout
table).  The table itself did not survive, so the byte order inside a tile is
taken from NVIDIA's public description of the block-scale-factor layout that
tcgen05 block-scaled MMA consumes (the same layout cuBLAS documents for 1D
block scaling): a 128-row x 4-column tile is 512 contiguous bytes, where row
r and column c of the tile land at

    (r % 32) * 16 + (r // 32) * 4 + c,

tiles are ordered row-block major (all column blocks of rows 0..127, then of
rows 128..255, ...), and the matrix is zero-padded to whole tiles.  This
reading is pinned by the GEMM parity tests: a wrong byte order feeds the
tensor cores the wrong scales.

Grouped forms (a reading, needed because each tcgen05 scale tile is a whole
128x4 tile and a GEMM tile must not mix experts):
* ``group_axis = 0`` (forward / dgrad: groups of rows): every group's first
  row starts a new 128-row block; the buffer has room for
  ``ceil(R/128) + E`` row blocks.
* ``group_axis = 1`` (wgrad: groups along the contracting dimension, whose
  32-element blocks are the scale columns): every group's first scale column
  starts a new 4-column block; the buffer has ``ceil(Cs/4) + E`` column
  blocks.
Unused bytes are zero.
"""
from __future__ import annotations

import numpy as np

from .quant import group_bounds, padded_starts

NO_GROUPS, GROUP_ROWS, GROUP_COLS = -1, 0, 1


def _cdiv(a, b):
    return (a + b - 1) // b


def swizzled_shape(R: int, Cs: int, E: int = 0, group_axis: int = NO_GROUPS):
    """(padded rows, padded columns) of one swizzled scale matrix."""
    rb, cb = _cdiv(R, 128), _cdiv(Cs, 4)
    if group_axis == GROUP_ROWS:
        rb += E
    elif group_axis == GROUP_COLS:
        cb += E
    return rb * 128, cb * 4


def tile_offset(r, c, padded_cols: int):
    """Byte offset of padded-matrix element (r, c) in the tiled layout."""
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    tile = (r // 128) * (padded_cols // 4) + c // 4
    return tile * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)


def swizzle(s, offs=None, group_axis: int = NO_GROUPS):
    """Swizzle ``s [R, Cs]`` (or batched ``[B, R, Cs]`` without groups).

    ``offs`` (cumulative exclusive ends) is over rows for ``GROUP_ROWS`` and
    over the *element* index of the contracting dimension (32 elements per
    scale column, boundaries multiples of 32) for ``GROUP_COLS``.
    Returns a flat uint8 array.
    """
    s = np.asarray(s, dtype=np.uint8)
    if s.ndim == 3:
        if group_axis != NO_GROUPS:
            raise ValueError("batched swizzle takes no groups")
        return np.concatenate([swizzle(s[b]) for b in range(s.shape[0])]) if s.shape[0] else \
            np.zeros(0, np.uint8)
    R, Cs = s.shape
    E = 0 if offs is None else len(offs)
    Rp, Cp = swizzled_shape(R, Cs, E, group_axis)
    out = np.zeros(Rp * Cp, dtype=np.uint8)
    rows = np.arange(R, dtype=np.int64)
    cols = np.arange(Cs, dtype=np.int64)
    if group_axis == GROUP_ROWS:
        starts, ends = group_bounds(offs)
        P = padded_starts(offs, 128)
        g = np.searchsorted(ends, rows, side="right")      # group of each row
        prow = P[g] + (rows - starts[g])
        pcol = cols
    elif group_axis == GROUP_COLS:
        offs = np.asarray(offs, dtype=np.int64)
        if np.any(offs % 32):
            raise ValueError("column groups must be multiples of 32 elements")
        sc_offs = offs // 32
        starts, ends = group_bounds(sc_offs)
        Q = padded_starts(sc_offs, 4)
        g = np.searchsorted(ends, cols, side="right")
        pcol = Q[g] + (cols - starts[g])
        prow = rows
    else:
        prow, pcol = rows, cols
    o = tile_offset(prow[:, None], pcol[None, :], Cp)
    out[o.ravel()] = s.ravel()
    return out


def unswizzle(buf, Rp: int, Cp: int):
    """Inverse of the tile map for a whole padded matrix: returns [Rp, Cp].

    Written from the byte position's point of view (tile number, then
    position inside the tile), independent of ``tile_offset``.
    """
    buf = np.asarray(buf, dtype=np.uint8)
    out = np.zeros((Rp, Cp), dtype=np.uint8)
    tiles_per_row_block = Cp // 4
    for o in range(Rp * Cp):
        tile, w = divmod(o, 512)
        rb, cb = divmod(tile, tiles_per_row_block)
        r32, rest = divmod(w, 16)
        rq, c4 = divmod(rest, 4)
        out[rb * 128 + rq * 32 + r32, cb * 4 + c4] = buf[o]
    return out
