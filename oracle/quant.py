"""Dynamic FP8 quantization, written out step by step (CPU oracle).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this file.

Rowwise / colwise FP8.  The pages describe one quantization as a chain of
steps: take the per-row (or per-column) absolute maximum, derive the scale,
apply it, clamp, cast to FP8 ("Az AMD GPU-kon is gyorsult az FP8-as
PyTorch-tréning", section "A Triton-kernelok csökkentették a kvantálás
költségét"; "FP8-обучение на AMD", section "Три уровня оптимизации
Triton-ядер").  Activations get row scales, expert weights get column scales
per expert, and a routing offsets tensor sends rows to experts
("FP8-обучение на AMD", section "MoE: почему DeepSeek-V3 ломал пайплайн").

The pages fix neither the scale formula nor the precision; the readings
taken here:
* arithmetic in fp32 (the kernel's precision, so that both sides take every
  rounding decision identically): amax = max|x| (exact for bf16 inputs),
  s = fl32(fp8_max / max(amax, 1e-12)), q = enc(fl32(x * s)),
  stored dequantization scale inv = fl32(1 / s);
* the 1e-12 floor makes an all-zero row (or an empty group) well defined;
* the scale is applied by multiplication, and is not rounded to a power of
  two.

MXFP8.  Blocks of 32 consecutive elements share one e8m0 scale and the data
is e4m3 ("Accelerating Llama4 Scout training with TorchAO MXFP8 MoE
primitives", MXFP8 data / scale layout diagram).  The scale exponent is
floor(log2(amax)) - 8, clamped (see ``formats.e8m0_from_amax``); the data is
enc_fn(x * 2^-e), computed exactly in float64.  ``dim0`` blocks run along the
contiguous (last) dimension; ``dim1`` blocks run along dimension -2 and the
output is written transposed, which is the operand layout the backward
GEMMs contract over ("...MXFP8 MoE primitives", section on forward/backward
quantization and the contracting dimension of the weight gradient).
"""
from __future__ import annotations

import numpy as np

from .formats import FN, FNUZ, FP8_MAX, encode, e8m0_from_amax

EPS = np.float32(1e-12)


def _f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float32)


def _scale_from_amax(amax: np.ndarray, kind: str):
    amax = _f32(amax)
    s = np.float32(FP8_MAX[kind]) / np.maximum(amax, EPS)   # fp32 divide
    inv = np.float32(1.0) / s                               # fp32 divide
    return s.astype(np.float32), inv.astype(np.float32)


# ----------------------------------------------------------------------------
# rowwise / colwise
# ----------------------------------------------------------------------------

def quantize_rowwise(x, kind: str = FN):
    """Per-row FP8 quantization of ``x [R, C]`` (bf16 values as float32).

    Returns ``(q uint8 [R, C], inv float32 [R])``.
    """
    x = _f32(x)
    R, C = x.shape
    if C == 0:
        return np.zeros((R, 0), np.uint8), _scale_from_amax(np.zeros(R, np.float32), kind)[1]
    amax = np.max(np.abs(x), axis=1)
    s, inv = _scale_from_amax(amax, kind)
    q = encode(x * s[:, None], kind)                      # fp32 multiply
    return q, inv


def quantize_tensorwise(x, kind: str = FN):
    """One FP8 scale for the whole tensor ``x`` (any shape, bf16 values as
    float32): the coarsest of the four scaling granularities the pages list
    ("FP8-обучение на AMD", section "Скейлы: от тензора до микроблока": one
    scale for the whole tensor).  The arithmetic is the rowwise one with the
    absolute maximum taken over every element.

    Returns ``(q uint8 [x.shape], inv float32 scalar)``.
    """
    x = _f32(x)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)
    s = np.float32(np.float32(FP8_MAX[kind]) / np.maximum(amax, EPS))   # fp32 divide
    inv = np.float32(np.float32(1.0) / s)                               # fp32 divide
    q = encode(x * s, kind)                                             # fp32 multiply
    return q, inv


def quantize_colwise_3d(x, kind: str = FN, transpose_out: bool = True):
    """Per-(expert, column) FP8 quantization of dense ``x [E, R, C]``.

    The absolute maximum runs over R for each (e, c).  Returns
    ``(q, inv [E, C])`` with ``q`` of shape ``[E, C, R]`` when
    ``transpose_out`` (R contiguous: the K-major operand of a GEMM that
    contracts over R) or ``[E, R, C]`` otherwise.
    """
    x = _f32(x)
    E, R, C = x.shape
    amax = np.max(np.abs(x), axis=1) if R else np.zeros((E, C), np.float32)
    s, inv = _scale_from_amax(amax, kind)
    q = encode(x * s[:, None, :], kind)
    if transpose_out:
        q = np.ascontiguousarray(q.transpose(0, 2, 1))
    return q, inv


def jagged_t_cols(M: int, E: int) -> int:
    """Width of the transposed jagged output: every group padded to 32.

    Group ``e`` occupies columns ``[P_e, P_e + g_e)`` with
    ``P_e = sum_{j<e} round_up(g_j, 32)``; the width is a fixed bound
    ``round_up(M + 31*E, 16)`` so that it does not depend on the offsets.
    Padding columns hold code 0.
    """
    return (M + 31 * E + 15) // 16 * 16


def group_bounds(offs):
    offs = np.asarray(offs, dtype=np.int64)
    starts = np.concatenate([[0], offs[:-1]]) if len(offs) else np.zeros(0, np.int64)
    return starts, offs


def padded_starts(offs, unit: int):
    """Start of each group after rounding every earlier group up to ``unit``."""
    starts, ends = group_bounds(offs)
    sizes = ends - starts
    padded = (sizes + unit - 1) // unit * unit
    return np.concatenate([[0], np.cumsum(padded)[:-1]]).astype(np.int64) if len(sizes) else padded


def check_offsets(offs, M: int, multiple: int = 1):
    starts, ends = group_bounds(offs)
    if len(ends) == 0 or ends[-1] != M or np.any(ends < starts) or np.any(starts < 0):
        raise ValueError("offsets must be non-decreasing with offs[E-1] == M")
    if multiple > 1 and np.any(ends % multiple):
        raise ValueError(f"group boundaries must be multiples of {multiple}")


def quantize_colwise_jagged(x, offs, kind: str = FN, transpose_out: bool = True):
    """Per-(group, column) FP8 quantization of routed rows ``x [M, C]``.

    Group ``e`` is rows ``[offs[e-1], offs[e])``.  Returns
    ``(q, inv [E, C])``; ``q`` is ``[C, jagged_t_cols(M, E)]`` with the
    group-padded column layout of ``jagged_t_cols`` when ``transpose_out``,
    else ``[M, C]``.  An empty group gets inv = fl32(1 / fl32(max / 1e-12)).
    """
    x = _f32(x)
    M, C = x.shape
    check_offsets(offs, M)
    starts, ends = group_bounds(offs)
    E = len(ends)
    inv = np.empty((E, C), np.float32)
    q = np.empty((M, C), np.uint8)
    for e in range(E):
        seg = x[starts[e]:ends[e]]
        amax = np.max(np.abs(seg), axis=0) if len(seg) else np.zeros(C, np.float32)
        s, inv[e] = _scale_from_amax(amax, kind)
        q[starts[e]:ends[e]] = encode(seg * s[None, :], kind)
    if not transpose_out:
        return q, inv
    W = jagged_t_cols(M, E)
    qt = np.zeros((C, W), np.uint8)
    P = padded_starts(offs, 32)
    for e in range(E):
        g = ends[e] - starts[e]
        qt[:, P[e]:P[e] + g] = q[starts[e]:ends[e]].T
    return qt, inv


# ----------------------------------------------------------------------------
# MXFP8
# ----------------------------------------------------------------------------

def mxfp8_quantize_dim0(x):
    """MXFP8 along the last dimension: ``x [..., C]`` with C % 32 == 0.

    Returns ``(q uint8 [..., C], scale e8m0 uint8 [..., C/32])``.
    """
    x = np.asarray(x, dtype=np.float64)
    C = x.shape[-1]
    if C % 32:
        raise ValueError("C must be a multiple of 32")
    blocks = x.reshape(x.shape[:-1] + (C // 32, 32))
    amax = np.max(np.abs(blocks), axis=-1) if C else np.zeros(x.shape[:-1] + (0,))
    sb = e8m0_from_amax(amax)
    e = sb.astype(np.int64) - 127
    y = blocks * np.ldexp(1.0, (-e).astype(np.int32))[..., None]   # exact
    q = encode(y, FN).reshape(x.shape)
    return q, sb


def mxfp8_quantize_dim1(x):
    """MXFP8 along dimension -2 of ``x [..., R, C]`` (R % 32 == 0).

    Output is transposed: ``(qt uint8 [..., C, R], scale uint8 [..., C, R/32])``.
    Written directly with blocks along axis -2 (not via ``dim0`` of a
    transpose, which the tests use as an independent check).
    """
    x = np.asarray(x, dtype=np.float64)
    R, C = x.shape[-2], x.shape[-1]
    if R % 32:
        raise ValueError("R must be a multiple of 32")
    lead = x.shape[:-2]
    blocks = x.reshape(lead + (R // 32, 32, C))
    amax = np.max(np.abs(blocks), axis=-2) if R else np.zeros(lead + (0, C))
    sb = e8m0_from_amax(amax)                               # [..., R/32, C]
    e = sb.astype(np.int64) - 127
    y = blocks * np.ldexp(1.0, (-e).astype(np.int32))[..., None, :]
    q = encode(y, FN).reshape(lead + (R, C))
    qt = np.ascontiguousarray(np.swapaxes(q, -1, -2))
    st = np.ascontiguousarray(np.swapaxes(sb, -1, -2))
    return qt, st


# ----------------------------------------------------------------------------
# dequantization (used by the GEMM oracle)
# ----------------------------------------------------------------------------

def dequant_mx(q, sb):
    """float64 value of MXFP8 data ``q [..., C]`` with scales ``sb [..., C/32]``."""
    from .formats import decode, e8m0_value
    v = decode(q, FN)
    sc = np.repeat(e8m0_value(sb), 32, axis=-1)
    return v * sc


def dequant_rows(q, inv, kind: str = FN):
    """float64 value of rowwise data ``q [R, C]`` with per-row ``inv [R]``."""
    from .formats import decode
    return decode(q, kind) * np.asarray(inv, np.float64)[..., :, None]
