"""Token routing into expert groups and back, written out directly (CPU oracle).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this file.

The pages route each token to a few experts and place the routed rows by an
offsets tensor before the fused quantization and the one-launch grouped GEMM
("FP8-обучение на AMD", section "MoE: почему DeepSeek-V3 ломал пайплайн":
tokens are routed by offsets; "Az AMD GPU-kon is gyorsult az FP8-as
PyTorch-tréning", MoE section: experts receive batches of varying size).
The layer configurations pad every expert's group to a multiple of 32 rows,
the MXFP8 block length.  Readings taken here:
* the rows of expert e are the (token t, slot j) pairs with idx[t, j] == e in
  increasing (t, j) order (a stable placement);
* group e starts at P_e = sum over e' < e of round_up(count_e', 32); its
  padding rows are zero; offs[e] = P_e + round_up(count_e, 32), except that
  the last group also takes the slack up to the buffer size
  round_up(T * k + 31 * E, 32), a bound known without reading the counts;
* permute may weight each routed row: bf16(fp32(w) * x) (round to nearest
  even);
* unpermute: out[t] = bf16(sum over j in order of fp32(w[t, j]) * y[row])
  with fp32 products and sums (w = 1 when absent).
"""
from __future__ import annotations

import numpy as np


def route_rows(T: int, k: int, E: int) -> int:
    """Rows of the grouped buffer: every group padded to 32, plus slack."""
    return (T * k + 31 * E + 31) // 32 * 32


def _bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest bf16 value (ties to even), as float32."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def route_permute(x, idx, E: int, w=None):
    """x [T, H] (bf16 values as float32), idx [T, k] int -> (a [Mr, H],
    offs [E] int32, row_of [T, k] int32)."""
    x = np.asarray(x, np.float32)
    idx = np.asarray(idx)
    T, k = idx.shape
    H = x.shape[1]
    Mr = route_rows(T, k, E)
    counts = np.zeros(E, np.int64)
    for t in range(T):
        for j in range(k):
            counts[idx[t, j]] += 1
    padded = (counts + 31) // 32 * 32
    starts = np.concatenate([[0], np.cumsum(padded)[:-1]])
    offs = starts + padded
    offs[-1] = Mr
    a = np.zeros((Mr, H), np.float32)
    row_of = np.zeros((T, k), np.int32)
    fill = starts.copy()
    for t in range(T):            # increasing (t, j): the stable order
        for j in range(k):
            e = idx[t, j]
            r = fill[e]
            fill[e] += 1
            row_of[t, j] = r
            a[r] = x[t] if w is None else _bf16_round(np.float32(w[t, j]) * x[t])
    return a, offs.astype(np.int32), row_of


def route_unpermute(y, row_of, w=None):
    """y [Mr, N] (bf16 values as float32), row_of [T, k] -> out [T, N] (bf16
    values as float32)."""
    y = np.asarray(y, np.float32)
    T, k = row_of.shape
    acc = np.zeros((T, y.shape[1]), np.float32)
    for j in range(k):
        term = y[row_of[:, j]]
        if w is not None:
            term = (np.asarray(w, np.float32)[:, j:j + 1] * term).astype(np.float32)
        acc = (acc + term).astype(np.float32)
    return _bf16_round(acc)
