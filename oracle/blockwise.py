"""Blockwise FP8 quantization: one scale per fixed-size tile (CPU oracle).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this file.

The pages list four scaling granularities, from one scale per tensor, over
one per row and one per tile of fixed size ("blockwise"), to MXFP8's scale
per 32-element group ("FP8-обучение на AMD", section "Скейлы: от тензора до
микроблока"; the glossary of the Korean summary of the same article names
tensorwise, rowwise and blockwise as the coarser strategies).  They give no
tile size and no formula.  Readings taken here:

* the arithmetic of a tile is the rowwise one (``quant.py``): in fp32,
  amax = max|x| over the tile, s = fl32(fp8_max / max(amax, 1e-12)),
  q = enc(fl32(x * s)), stored dequantization scale inv = fl32(1 / s);
* activations and gradients (the row operand of forward and dgrad) use
  1 x 128 tiles along the contracting (last) dimension; expert weights use
  128 x 128 tiles, so that one set of weight scales serves the forward
  (contracting over K) and the transposed weight of dgrad (contracting over
  N);
* the operands of wgrad (dY and A, contracting over the routed tokens) use
  128 x 1 tiles along the tokens, cut per group: block j of group e is
  tokens [start_e + 128 j, min(end_e, start_e + 128 (j + 1))), so a group's
  last block may be shorter; group boundaries are multiples of 32 (the MoE
  layers pad every group to 32 rows);
* dense dimensions that carry tiles are multiples of 128;
* scale layouts (fp32): row tiles of x [R, C] -> inv [C/128, R] (tile index
  major: the 128 row scales of one tile column are contiguous); weight tiles
  of w [E, N, K] -> inv [E, N/128, K/128]; token tiles of x [M, C] ->
  inv [n_blocks, C] with the blocks of all groups in order.
"""
from __future__ import annotations

import numpy as np

from .formats import FN, FP8_MAX, decode, encode
from .quant import check_offsets, group_bounds

TILE = 128
EPS = np.float32(1e-12)


def _scale(amax, kind):
    amax = np.asarray(amax, np.float32)
    s = (np.float32(FP8_MAX[kind]) / np.maximum(amax, EPS)).astype(np.float32)   # fp32 divide
    inv = (np.float32(1.0) / s).astype(np.float32)                                 # fp32 divide
    return s, inv


def quantize_blockwise_rows(x, kind: str = FN):
    """1 x 128 tiles along the last dimension of ``x [R, C]`` (C % 128 == 0).

    Returns ``(q uint8 [R, C], inv float32 [C/128, R])``.
    """
    x = np.asarray(x, np.float32)
    R, C = x.shape
    if C % TILE:
        raise ValueError("C must be a multiple of 128")
    nb = C // TILE
    inv = np.empty((nb, R), np.float32)
    q = np.empty((R, C), np.uint8)
    for b in range(nb):
        tile = x[:, b * TILE:(b + 1) * TILE]
        amax = np.max(np.abs(tile), axis=1) if R else np.zeros(0, np.float32)
        s, inv[b] = _scale(amax, kind)
        q[:, b * TILE:(b + 1) * TILE] = encode(tile * s[:, None], kind)    # fp32 multiply
    return q, inv


def quantize_blockwise_weight(w, kind: str = FN):
    """128 x 128 tiles of expert weights ``w [E, N, K]`` (N, K % 128 == 0).

    Returns ``(q uint8 [E, N, K], inv float32 [E, N/128, K/128])``; the
    transposed codes of the dgrad operand are ``q.transpose(0, 2, 1)`` with
    the same scales (tile (nb, kb) of W is tile (kb, nb) of W^T).
    """
    w = np.asarray(w, np.float32)
    E, N, K = w.shape
    if N % TILE or K % TILE:
        raise ValueError("N and K must be multiples of 128")
    inv = np.empty((E, N // TILE, K // TILE), np.float32)
    q = np.empty((E, N, K), np.uint8)
    for e in range(E):
        for nb in range(N // TILE):
            for kb in range(K // TILE):
                tile = w[e, nb * TILE:(nb + 1) * TILE, kb * TILE:(kb + 1) * TILE]
                s, inv[e, nb, kb] = _scale(np.max(np.abs(tile)), kind)
                q[e, nb * TILE:(nb + 1) * TILE, kb * TILE:(kb + 1) * TILE] = encode(tile * s, kind)
    return q, inv


def token_blocks(offs):
    """Token tiles of the groups: list of (group, start, end) in block order."""
    starts, ends = group_bounds(offs)
    out = []
    for e in range(len(ends)):
        for b0 in range(int(starts[e]), int(ends[e]), TILE):
            out.append((e, b0, min(int(ends[e]), b0 + TILE)))
    return out


def quantize_blockwise_tokens(x, offs, kind: str = FN):
    """128 x 1 tiles along the routed tokens of ``x [M, C]``, cut per group
    (offsets multiples of 32), output transposed.

    Returns ``(qt uint8 [C, M], inv float32 [n_blocks, C])``: column m of
    ``qt`` holds token m (the operand layout of wgrad, tokens contiguous).
    """
    x = np.asarray(x, np.float32)
    M, C = x.shape
    check_offsets(offs, M, 32)
    blocks = token_blocks(offs)
    inv = np.empty((len(blocks), C), np.float32)
    q = np.empty((M, C), np.uint8)
    for i, (_, b0, b1) in enumerate(blocks):
        tile = x[b0:b1]
        s, inv[i] = _scale(np.max(np.abs(tile), axis=0), kind)
        q[b0:b1] = encode(tile * s[None, :], kind)
    return np.ascontiguousarray(q.T), inv


# ----------------------------------------------------------------------------
# dequantization (operands of the GEMM oracle)
# ----------------------------------------------------------------------------

def dequant_rows(q, inv, kind: str = FN):
    """float64 value of 1 x 128-tiled ``q [R, C]`` with ``inv [C/128, R]``."""
    v = decode(q, kind)
    return v * np.repeat(np.asarray(inv, np.float64).T, TILE, axis=1)


def dequant_weight(q, inv, kind: str = FN):
    """float64 value of 128 x 128-tiled ``q [E, N, K]`` with ``inv [E, N/128, K/128]``."""
    v = decode(q, kind)
    sc = np.repeat(np.repeat(np.asarray(inv, np.float64), TILE, axis=1), TILE, axis=2)
    return v * sc


def dequant_tokens(qt, inv, offs, kind: str = FN):
    """float64 value of token-tiled ``qt [C, M]`` with ``inv [n_blocks, C]``."""
    v = decode(qt, kind)
    out = np.empty_like(v)
    for i, (_, b0, b1) in enumerate(token_blocks(offs)):
        out[:, b0:b1] = v[:, b0:b1] * np.asarray(inv[i], np.float64)[:, None]
    return out
