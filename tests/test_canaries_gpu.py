"""Every C-ABI call writes inside its output buffers only: each output is a
view into a larger allocation whose 256 bytes before and 4 KB after hold a
canary pattern, checked unchanged after the call (ragged shapes, so that
tails and padding paths run)."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
LEAD, TAIL, PAT = 256, 4096, 0xA5


@pytest.fixture(scope="module")
def F():
    from mxfp8_moe_quantization_gb300 import build as B
    B.build()
    import mxfp8_moe_quantization_gb300 as m
    return m


class Guarded:
    """Output buffers carved out of canary-filled allocations."""

    def __init__(self):
        self.bufs = []

    def __call__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((LEAD + n + TAIL,), PAT, dtype=torch.uint8, device=DEV)
        self.bufs.append((raw, n))
        return raw[LEAD:LEAD + n].view(dtype).view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        for raw, n in self.bufs:
            lead = raw[:LEAD]
            tail = raw[LEAD + n:]
            assert bool((lead == PAT).all()) and bool((tail == PAT).all()), f"{what}: write outside an output buffer"
        self.bufs.clear()


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16).to(DEV)


def test_quantization_outputs_stay_in_bounds(F):
    g = Guarded()
    u8, f32 = torch.uint8, torch.float32
    x = _bf16((77, 160), 1)
    for kind in (F.E4M3FN, F.E4M3FNUZ):
        F.fp8moe_quantize_rowwise(x, kind, q=g((77, 160), u8), scale_inv=g((77,), f32))
    g.check("rowwise")
    w = _bf16((3, 48, 160), 2)
    F.fp8moe_quantize_colwise_3d(w, None, True, q=g((3, 160, 48), u8), scale_inv=g((3, 160), f32))
    F.fp8moe_quantize_colwise_3d(w, None, False, q=g((3, 48, 160), u8), scale_inv=g((3, 160), f32))
    sizes = [30, 0, 47]
    offs = torch.from_numpy(W.offsets_from_sizes(sizes)).to(DEV)
    xj = _bf16((77, 48), 3)
    F.fp8moe_quantize_colwise_3d(xj, offs, True, q=g((48, F.fp8moe_jagged_t_cols(77, 3)), u8),
                                 scale_inv=g((3, 48), f32))
    g.check("colwise")
    F.fp8moe_quantize_tensorwise(x, q=g((77, 160), u8), scale_inv=g((1,), f32))
    F.fp8moe_quantize_tensorwise(xj, offs, True, q=g((48, F.fp8moe_jagged_t_cols(77, 3)), u8),
                                 scale_inv=g((1,), f32))
    g.check("tensorwise")
    xm = _bf16((96, 160), 4)
    F.fp8moe_mxfp8_quantize_dim0(xm, q=g((96, 160), u8), scale=g((96, 5), u8))
    F.fp8moe_mxfp8_quantize_dim1(xm, qt=g((160, 96), u8), scale=g((160, 3), u8))
    s_rm = torch.empty(96, 5, dtype=u8, device=DEV)
    F.fp8moe_mxfp8_quantize_dim0(xm, scale=s_rm)
    F.fp8moe_swizzle_scales_128x4(s_rm, out=g((F.fp8moe_swizzled_scales_bytes(1, 96, 5, 0, F.NO_GROUPS),), u8))
    g.check("mxfp8 dim0 / dim1 / swizzle")
    offs_m = torch.from_numpy(W.offsets_from_sizes([32, 0, 64])).to(DEV)
    F.fp8moe_mxfp8_quantize_dual(
        xm, offs_m, F.GROUP_ROWS, F.GROUP_COLS, q0=g((96, 160), u8),
        s0=g((F.fp8moe_swizzled_scales_bytes(1, 96, 5, 3, F.GROUP_ROWS),), u8), q1=g((160, 96), u8),
        s1=g((F.fp8moe_swizzled_scales_bytes(1, 160, 3, 3, F.GROUP_COLS),), u8))
    g.check("dual")
    xb = _bf16((37, 384), 5)
    F.fp8moe_quantize_blockwise_rows(xb, q=g((37, 384), u8), scale_inv=g((3, 37), f32))
    wb = _bf16((2, 256, 128), 6)
    F.fp8moe_quantize_blockwise_weight(wb, q=g((2, 256, 128), u8), qt=g((2, 128, 256), u8),
                                       scale_inv=g((2, 2, 1), f32))
    xt = _bf16((96, 48), 7)
    F.fp8moe_quantize_blockwise_tokens(xt, offs_m, qt=g((48, 96), u8),
                                       scale_inv=g((F.fp8moe_blockwise_token_blocks(96, 3), 48), f32))
    g.check("blockwise")
    assert F.fp8moe_get_device_status() == 0


def test_gemm_and_routing_outputs_stay_in_bounds(F):
    g = Guarded()
    bf = torch.bfloat16
    sizes = [64, 0, 96, 32]
    offs = torch.from_numpy(W.offsets_from_sizes(sizes)).to(DEV)
    M, E, N, K = 192, 4, 288, 256            # N: one full and one partial 256-column tile
    codes = lambda *s: torch.randint(0, 120, s, dtype=torch.uint8, device=DEV)
    one = lambda n: torch.full((n,), 127, dtype=torch.uint8, device=DEV)
    qa, qw, qdy, qwt, qdyt, qat = codes(M, K), codes(E, N, K), codes(M, N), codes(E, K, N), codes(N, M), codes(K, M)
    sa = one(F.fp8moe_swizzled_scales_bytes(1, M, K // 32, E, F.GROUP_ROWS))
    sw = one(F.fp8moe_swizzled_scales_bytes(E, N, K // 32))
    sdy = one(F.fp8moe_swizzled_scales_bytes(1, M, N // 32, E, F.GROUP_ROWS))
    swt = one(F.fp8moe_swizzled_scales_bytes(E, K, N // 32))
    sdyt = one(F.fp8moe_swizzled_scales_bytes(1, N, M // 32, E, F.GROUP_COLS))
    sat = one(F.fp8moe_swizzled_scales_bytes(1, K, M // 32, E, F.GROUP_COLS))
    F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, qa, sa, qw, sw, offs, out=g((M, N), bf))
    F.fp8moe_scaled_grouped_mm_dgrad(F.MXFP8, qdy, sdy, qwt, swt, offs, out=g((M, K), bf))
    F.fp8moe_scaled_grouped_mm_wgrad(F.MXFP8, qdyt, sdyt, qat, sat, offs, M, out=g((E, N, K), bf))
    g.check("MXFP8 GEMMs")
    ones = lambda *s: torch.ones(s, dtype=torch.float32, device=DEV)
    Mt = F.fp8moe_jagged_t_cols(M, E)
    F.fp8moe_scaled_grouped_mm_fwd(F.ROWWISE, qa, ones(M), qw, ones(E, N), offs, out=g((M, N), bf))
    F.fp8moe_scaled_grouped_mm_wgrad(F.ROWWISE, codes(N, Mt), ones(E, N), codes(K, Mt), ones(E, K), offs, M,
                                     out=g((E, N, K), bf))
    g.check("rowwise GEMMs")
    Nb = 384
    qwb, qdyb = codes(E, Nb, K), codes(M, Nb)
    F.fp8moe_scaled_grouped_mm_fwd(F.BLOCKWISE, qa, ones(K // 128, M), qwb, ones(E, Nb // 128, K // 128), offs,
                                   out=g((M, Nb), bf))
    nblk = F.fp8moe_blockwise_token_blocks(M, E)
    F.fp8moe_scaled_grouped_mm_wgrad(F.BLOCKWISE, codes(Nb, M), ones(nblk, Nb), qat, ones(nblk, K), offs, M,
                                     out=g((E, Nb, K), bf))
    g.check("blockwise GEMMs")
    T, k, H = 50, 2, 64
    x = _bf16((T, H), 8)
    idx = torch.randint(0, E, (T, k), dtype=torch.int32, device=DEV)
    rows = F.fp8moe_route_rows(T, k, E)
    a, o, row_of = F.fp8moe_route_permute(x, idx, E, a=g((rows, H), bf), offs=g((E,), torch.int32),
                                          row_of=g((T, k), torch.int32))
    F.fp8moe_route_unpermute(a, row_of, out=g((T, H), bf))
    g.check("routing")
    a2, w2, dy2 = _bf16((M, K), 9), _bf16((E, 256, K), 10, 0.05), _bf16((M, 256), 11)
    ws = g((F.fp8moe_mxfp8_moe_workspace_bytes(E, M, 256, K),), torch.uint8)
    F.fp8moe_mxfp8_moe_fwd(a2, w2, offs, workspace=ws, out=g((M, 256), bf))
    F.fp8moe_mxfp8_moe_bwd(dy2, offs, ws, K, da=g((M, K), bf), dw=g((E, 256, K), bf))
    g.check("layer composites")
    assert F.fp8moe_get_device_status() == 0
