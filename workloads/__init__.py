"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module only draws random numbers and lays them out: it holds none of the
quantization or GEMM arithmetic.  Both sides (the CUDA library and the CPU
oracle) receive the tensors it returns as inputs.

Shapes and distributions follow the five workloads the FP8/MXFP8 MoE pages
discuss (see "FP8 Training on AMD GPUs with TorchTitan and TorchAO" and
"Accelerating Llama4 Scout training with TorchAO MXFP8 MoE primitives"):

* ``tiny``        E=4, K=256, N=512, M=1024, Dirichlet(0.5) groups in units of
                  32 with one group forced empty, 2% of rows scaled x100.
* ``llama3_8b``   dense linear, X [8192,4096] N(0,1) with 0.1% elements x50,
                  W [14336,4096] N(0,0.02).
* ``dsmoe_16b``   64 experts, hidden 2048, FFN 1408, 8192 tokens top-6,
                  Zipf(1.1) expert popularity (rowwise FP8).
* ``scout``       16 experts, hidden 5120, FFN 8192, 16384 tokens top-1,
                  Dirichlet(1) loads padded to multiples of 32, 0.5% x30
                  outliers (MXFP8).
* ``dsv3``        256 experts, hidden 7168, FFN 2048, 4096 tokens top-8,
                  Zipf(1.2) with 8 experts masked empty, padded to 32 (MXFP8).

Group layout: ``offs[e]`` is the exclusive end row of group ``e`` (a
cumulative sum), so group ``e`` is rows ``[offs[e-1], offs[e])`` with
``offs[-1] = 0``.  Padding rows (when a config pads groups to 32) are zero
rows placed after each group's real rows.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Tuple

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "get_workload", "group_sizes", "offsets_from_sizes",
    "bf16_bits_from_f32", "make_bf16", "make_activations", "make_weights",
]


# ----------------------------------------------------------------------------
# routing / group sizes (host, numpy)
# ----------------------------------------------------------------------------

def _largest_remainder(p: np.ndarray, total: int) -> np.ndarray:
    """Integer counts proportional to ``p`` that sum exactly to ``total``."""
    raw = p * total
    base = np.floor(raw).astype(np.int64)
    rem = total - int(base.sum())
    order = np.argsort(-(raw - base), kind="stable")
    base[order[:rem]] += 1
    return base


def _dirichlet_units(rng: np.random.Generator, E: int, alpha: float, M: int,
                     unit: int, forced_zero: bool) -> np.ndarray:
    n_live = E - 1 if forced_zero else E
    p = rng.dirichlet([alpha] * n_live)
    units = _largest_remainder(p, M // unit) * unit
    if forced_zero:
        pos = int(rng.integers(0, E))
        units = np.insert(units, pos, 0)
    return units.astype(np.int64)


def _zipf_topk_counts(rng: np.random.Generator, E: int, T: int, k: int, s: float,
                      masked: int = 0) -> np.ndarray:
    """Token->expert histogram for top-k routing with Zipf(s) popularity.

    Experts get weight rank^-s over a seeded permutation; each token picks k
    distinct experts by Gumbel-top-k on the log-weights.  ``masked`` experts
    (seeded) receive no tokens.
    """
    perm = rng.permutation(E)
    w = np.empty(E)
    w[perm] = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    logw = np.log(w)
    if masked:
        dead = rng.choice(E, size=masked, replace=False)
        logw[dead] = -np.inf
    counts = np.zeros(E, dtype=np.int64)
    chunk = 4096
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        g = rng.gumbel(size=(t1 - t0, E))
        top = np.argpartition(-(logw[None, :] + g), k - 1, axis=1)[:, :k]
        counts += np.bincount(top.ravel(), minlength=E)
    return counts


def _multinomial_dirichlet(rng: np.random.Generator, E: int, T: int, alpha: float) -> np.ndarray:
    p = rng.dirichlet([alpha] * E)
    return rng.multinomial(T, p).astype(np.int64)


def _round_up(x, m):
    return (x + m - 1) // m * m


def offsets_from_sizes(sizes) -> np.ndarray:
    """Cumulative exclusive-end offsets (int32) from per-group sizes."""
    return np.cumsum(np.asarray(sizes, dtype=np.int64)).astype(np.int32)


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    recipe: str            # "mxfp8" or "rowwise"
    E: int                 # experts (1 for the dense linear)
    K: int                 # hidden (contracting dim of the forward GEMM)
    N: int                 # expert FFN / output features
    tokens: int
    topk: int
    description: str

    # ------------------------------------------------------------------
    def group_plan(self) -> Tuple[np.ndarray, np.ndarray]:
        """(real_counts[E], padded_sizes[E]) for this workload's routing."""
        rng = np.random.Generator(np.random.PCG64(self.seed))
        if self.name == "tiny":
            sizes = _dirichlet_units(rng, self.E, 0.5, self.tokens, 32, forced_zero=True)
            return sizes.copy(), sizes
        if self.name == "llama3_8b":
            s = np.array([self.tokens], dtype=np.int64)
            return s, s
        if self.name == "dsmoe_16b":
            c = _zipf_topk_counts(rng, self.E, self.tokens, self.topk, 1.1)
            return c, c
        if self.name == "scout":
            c = _multinomial_dirichlet(rng, self.E, self.tokens * self.topk, 1.0)
            return c, _round_up(c, 32)
        if self.name == "dsv3":
            c = _zipf_topk_counts(rng, self.E, self.tokens, self.topk, 1.2, masked=8)
            return c, _round_up(c, 32)
        raise KeyError(self.name)

    def offs(self) -> np.ndarray:
        return offsets_from_sizes(self.group_plan()[1])

    @property
    def M(self) -> int:
        return int(self.group_plan()[1].sum())


WORKLOADS: Dict[str, Workload] = {
    w.name: w for w in [
        Workload("tiny", 1001, "mxfp8", 4, 256, 512, 1024, 1,
                 "tiny MXFP8 MoE: E=4 K=256 N=512 M=1024, Dirichlet(0.5) groups of 32s, one empty"),
        Workload("llama3_8b", 1002, "rowwise", 1, 4096, 14336, 8192, 1,
                 "dense rowwise FP8 linear, Llama3-8B bs1 seq8192: X[8192,4096] W[14336,4096]"),
        Workload("dsmoe_16b", 1003, "rowwise", 64, 2048, 1408, 8192, 6,
                 "DeepSeek-MoE-16B rowwise FP8 grouped GEMM: 64 experts, 2048->1408, top-6 Zipf(1.1)"),
        Workload("scout", 1004, "mxfp8", 16, 5120, 8192, 16384, 1,
                 "Llama4-Scout MXFP8 grouped GEMM: 16 experts, 5120->8192, top-1 Dirichlet(1) padded to 32"),
        Workload("dsv3", 1005, "mxfp8", 256, 7168, 2048, 4096, 8,
                 "DeepSeek-V3 MoE layer MXFP8: 256 experts, 7168->2048, top-8 Zipf(1.2), 8 empty, padded to 32"),
    ]
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]


def group_sizes(name: str) -> np.ndarray:
    return WORKLOADS[name].group_plan()[1]


# ----------------------------------------------------------------------------
# tensors (torch: host or device; the caller picks the device)
# ----------------------------------------------------------------------------

def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16, returned as uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def make_bf16(shape, seed: int, std: float = 1.0, outlier_frac: float = 0.0,
              outlier_scale: float = 1.0, row_outliers: bool = False,
              zero_rows: Optional[np.ndarray] = None, device="cpu"):
    """bf16 N(0, std^2) tensor with optional outliers (torch, on ``device``).

    ``row_outliers``: the outlier mask selects whole rows (last dim kept).
    ``zero_rows``: boolean mask over dim 0 of rows to zero (group padding).
    """
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if outlier_frac > 0:
        mshape = shape[:-1] + (1,) if row_outliers else shape
        m = torch.rand(*mshape, generator=g, device=device) < outlier_frac
        x = torch.where(m, x * outlier_scale, x)
    if zero_rows is not None:
        zr = torch.as_tensor(zero_rows, device=device).reshape(-1, *([1] * (len(shape) - 1)))
        x = x.masked_fill(zr, 0.0)
    return x.to(torch.bfloat16)


def padding_row_mask(wl: Workload) -> np.ndarray:
    """True for the zero rows a workload appends to each group (padding to 32)."""
    real, padded = wl.group_plan()
    mask = np.zeros(int(padded.sum()), dtype=bool)
    start = 0
    for r, p in zip(real, padded):
        mask[start + r:start + p] = True
        start += p
    return mask


def make_activations(wl: Workload, which: str, device="cpu"):
    """Routed activations ``A [M,K]`` or upstream gradient ``dY [M,N]``.

    ``which`` in {"A", "dY", "A2", "dY2"}: A/dY feed the first expert weight
    (``W1 [E,N,K]``); A2/dY2 feed the second (``W2 [E,K,N]``), standing in
    for the hidden activation and the layer-output gradient.
    """
    M = wl.M
    zero = padding_row_mask(wl)
    zero = zero if zero.any() else None
    cols = {"A": wl.K, "dY": wl.N, "A2": wl.N, "dY2": wl.K}[which]
    seed = wl.seed * 100 + {"A": 1, "dY": 2, "A2": 3, "dY2": 4}[which]
    if which.startswith("dY"):
        return make_bf16((M, cols), seed, 1.0, zero_rows=zero, device=device)
    if wl.name == "tiny":
        return make_bf16((M, cols), seed, 1.0, 0.02, 100.0, row_outliers=True,
                         zero_rows=zero, device=device)
    if wl.name == "llama3_8b":
        return make_bf16((M, cols), seed, 1.0, 0.001, 50.0, zero_rows=zero, device=device)
    if wl.name == "scout":
        return make_bf16((M, cols), seed, 1.0, 0.005, 30.0, zero_rows=zero, device=device)
    return make_bf16((M, cols), seed, 1.0, zero_rows=zero, device=device)


def make_weights(wl: Workload, which: str = "W1", device="cpu"):
    """Expert weights in nn.Linear layout: W1 ``[E,N,K]``, W2 ``[E,K,N]``."""
    shape = (wl.E, wl.N, wl.K) if which == "W1" else (wl.E, wl.K, wl.N)
    seed = wl.seed * 100 + (11 if which == "W1" else 12)
    return make_bf16(shape, seed, 0.02, device=device)
