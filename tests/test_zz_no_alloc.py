"""The routing permute without a caller workspace (fp8moe_route_permute_noalloc).

Some callers cannot allocate device memory when they route: a runtime that
plans all of its device memory up front into a fixed arena, or code on a
path where cudaMalloc is not allowed.  This entry point routes through the
library's own static scratch instead of a workspace the caller passes.  The
GPU test calls it through the C ABI twice in a row (different inputs, so a
second call that read what the first left in the shared scratch would show)
and compares each result with the workspace entry point's, bit for bit: the
routing is integer and copy work, so the two must be identical.

This file is collected last on purpose (its name sorts last).
"""
import ctypes

import numpy as np
import pytest
import torch

DEV = "cuda"


@pytest.fixture(scope="module")
def F():
    from mxfp8_moe_quantization_gb300 import build as B
    B.build()
    import mxfp8_moe_quantization_gb300 as m
    return m


def _case(T, k, E, H, seed):
    rng = np.random.default_rng(seed)
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.2
    p /= p.sum()
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    return x, idx, w


@pytest.mark.gpu
def test_noalloc_permute_matches_workspace_permute(F):
    lib = F.lib()
    cases = [(4096, 8, 256, 256, 1), (1500, 2, 16, 136, 2)]   # two calls in a row, different shapes
    for T, k, E, H, seed in cases:
        x, idx, w = _case(T, k, E, H, seed)
        xd, idxd, wd = x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(w).to(DEV)
        ref_a, ref_offs, ref_row = F.fp8moe_route_permute(xd, idxd, E, wd)
        rows = F.fp8moe_route_rows(T, k, E)
        # outputs preset to a pattern, so that a row the call fails to write shows
        a = torch.full((rows, H), 7.0, dtype=torch.bfloat16, device=DEV)
        offs = torch.full((E,), -3, dtype=torch.int32, device=DEV)
        row_of = torch.full((T, k), -3, dtype=torch.int32, device=DEV)
        stream = torch.cuda.current_stream().cuda_stream
        st = lib.fp8moe_route_permute_noalloc(xd.data_ptr(), T, H, idxd.data_ptr(), wd.data_ptr(), k, E,
                                              a.data_ptr(), offs.data_ptr(), row_of.data_ptr(), stream)
        assert st == 0, lib.fp8moe_status_string(st)
        assert F.fp8moe_get_device_status() == 0
        assert torch.equal(offs, ref_offs)
        assert torch.equal(row_of, ref_row)
        assert torch.equal(a.view(torch.int16), ref_a.view(torch.int16))


def test_noalloc_permute_rejects_problems_beyond_the_scratch():
    """A problem whose scratch exceeds the static array is refused on the
    host, before any CUDA call (no GPU needed)."""
    from mxfp8_moe_quantization_gb300 import build as B
    B.build()
    import mxfp8_moe_quantization_gb300 as F
    lib = F.lib()
    p = ctypes.c_void_p(1 << 20)
    T, k, E = 1 << 20, 8, 1024                      # 8 Mi (token, slot) pairs over 1024 experts
    assert lib.fp8moe_route_workspace_bytes(T, k, E) > F.ROUTE_STATIC_SCRATCH_BYTES
    assert lib.fp8moe_route_permute_noalloc(p, T, 64, p, None, k, E, p, p, p, None) == 7
    assert b"scratch" in lib.fp8moe_status_string(7)
