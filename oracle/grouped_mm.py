"""Scaled grouped GEMM for MoE, forward / dgrad / wgrad (CPU oracle).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this file.

What the pages fix: a MoE layer multiplies a 2D tensor of routed token rows
by a 3D tensor of expert weights, rows being assigned to experts by an
offsets tensor, in one grouped launch ("Accelerating Llama4 Scout training
with TorchAO MXFP8 MoE primitives", MoE forward diagram caption;
"FP8-обучение на AMD", section "MoE: почему DeepSeek-V3 ломал пайплайн");
each linear layer has three GEMMs -- forward, gradient w.r.t. the input,
gradient w.r.t. the weight ("FP8-обучение на AMD", section "Что такое
FP8-обучение"; "Az AMD GPU-kon ...", section "Az AMD FP8-formátumának
támogatása"); the weight gradient contracts over the routed-token dimension
("...MXFP8 MoE primitives", section details).

Definitions (operands already dequantized to float64 -- the value of each
FP8 code times its scale, both exact in float64 -- and accumulated in
float64; group e = rows / tokens ``[offs[e-1], offs[e])``):

    forward  out[m, :]  = A[m, :] @ W[e].T          A [M,K], W [E,N,K] -> [M,N]
    dgrad    dA[m, :]   = dY[m, :] @ Wt[e].T        dY [M,N], Wt [E,K,N] -> [M,K]
    wgrad    dW[e]      = dYt[:, grp] @ At[:, grp].T  dYt [N,M'], At [K,M'] -> [E,N,K]

Readings: an empty group contributes no rows to forward/dgrad and gives
dW[e] = 0 in wgrad; rows not covered by the offsets (offs[E-1] != M) are an
error.  For wgrad the token columns of group e are ``[col0[e], col0[e]+g_e)``:
the unpadded offsets for MXFP8 operands, the 32-padded starts for the
group-padded rowwise layout.

Each function also returns the elementwise bound sum_k |a_k b_k| used by the
GEMM tolerance.
"""
from __future__ import annotations

import numpy as np

from .quant import check_offsets, group_bounds


def grouped_mm_fwd(a, w, offs):
    a = np.asarray(a, np.float64)
    w = np.asarray(w, np.float64)
    M = a.shape[0]
    check_offsets(offs, M)
    starts, ends = group_bounds(offs)
    out = np.zeros((M, w.shape[1]))
    bound = np.zeros_like(out)
    for e in range(len(ends)):
        s, t = starts[e], ends[e]
        if t > s:
            out[s:t] = a[s:t] @ w[e].T
            bound[s:t] = np.abs(a[s:t]) @ np.abs(w[e]).T
    return out, bound


def grouped_mm_dgrad(dy, wt, offs):
    """Same contraction as forward, over the output-feature dimension."""
    return grouped_mm_fwd(dy, wt, offs)


def grouped_mm_wgrad(dyt, at, offs, col0=None):
    dyt = np.asarray(dyt, np.float64)
    at = np.asarray(at, np.float64)
    starts, ends = group_bounds(offs)
    if col0 is None:
        col0 = starts
    E = len(ends)
    out = np.zeros((E, dyt.shape[0], at.shape[0]))
    bound = np.zeros_like(out)
    for e in range(E):
        g = ends[e] - starts[e]
        if g > 0:
            c = slice(col0[e], col0[e] + g)
            out[e] = dyt[:, c] @ at[:, c].T
            bound[e] = np.abs(dyt[:, c]) @ np.abs(at[:, c]).T
    return out, bound


def brute_force_mm(a, b):
    """Triple-loop a @ b.T for tiny inputs (a pin for the library matmul)."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    out = np.zeros((a.shape[0], b.shape[0]))
    for i in range(a.shape[0]):
        for j in range(b.shape[0]):
            acc = 0.0
            for k in range(a.shape[1]):
                acc += a[i, k] * b[j, k]
            out[i, j] = acc
    return out
