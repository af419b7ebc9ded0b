"""GPU parity of the MXFP8 MoE layer composites (forward: dual quantization of
A and W + grouped GEMM forward; backward: dual quantization of dY + dgrad and
wgrad on the operands the forward kept).

* Against the CPU oracle chain (MXFP8 quantization of each operand along the
  contracting dimension of its GEMM, then the float64 grouped GEMM), with the
  grouped GEMM tolerance |gpu - ref| <= 8e-3 |ref| + 1e-3 sum_k |a_k b_k|.
* Bit-identical to the same chain of single calls through the C ABI, also at
  the Llama4-Scout layer size.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import grouped_mm as OG, quant as OQ

pytestmark = pytest.mark.gpu
DEV = "cuda"
RTOL, BTOL = 8e-3, 1e-3


@pytest.fixture(scope="module")
def F():
    from mxfp8_moe_quantization_gb300 import build as B
    B.build()
    import mxfp8_moe_quantization_gb300 as m
    return m


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


def _np(t):
    return t.float().cpu().numpy()


def _check(out, ref, bound, what):
    got = _np(out)
    err = np.abs(got - ref)
    lim = RTOL * np.abs(ref) + BTOL * bound
    assert np.all(err <= lim), f"{what}: worst excess {float((err - lim).max())}"


def _chain(F, a, w, dy, offs):
    """The composite's steps as single calls."""
    qa, sa, qat, sat = F.fp8moe_mxfp8_quantize_dual(a, offs, F.GROUP_ROWS, F.GROUP_COLS)
    qw, sw, qwt, swt = F.fp8moe_mxfp8_quantize_dual(w, None, F.NO_GROUPS, F.NO_GROUPS)
    out = F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, qa, sa, qw, sw, offs)
    qdy, sdy, qdyt, sdyt = F.fp8moe_mxfp8_quantize_dual(dy, offs, F.GROUP_ROWS, F.GROUP_COLS)
    da = F.fp8moe_scaled_grouped_mm_dgrad(F.MXFP8, qdy, sdy, qwt, swt, offs)
    dw = F.fp8moe_scaled_grouped_mm_wgrad(F.MXFP8, qdyt, sdyt, qat, sat, offs, a.shape[0])
    return out, da, dw


@pytest.mark.parametrize("sizes,N,K", [([64, 0, 352, 32, 160], 320, 384), ([0, 96, 0], 256, 64),
                                       ([224, 32], 32, 1024)])
def test_layer_against_oracle(F, sizes, N, K):
    offs = W.offsets_from_sizes(sizes)
    M, E = int(sum(sizes)), len(sizes)
    a = _bf16((M, K), 71, 1.0)
    w = _bf16((E, N, K), 72, 0.05)
    dy = _bf16((M, N), 73, 1.0)
    d_offs = torch.from_numpy(offs).to(DEV)
    out, ws = F.fp8moe_mxfp8_moe_fwd(a.to(DEV), w.to(DEV), d_offs)
    da, dw = F.fp8moe_mxfp8_moe_bwd(dy.to(DEV), d_offs, ws, K)
    assert F.fp8moe_get_device_status() == 0
    an, wn, dyn = _np(a), _np(w), _np(dy)
    # forward: A and W along K
    qa, sa = OQ.mxfp8_quantize_dim0(an)
    qw, sw = OQ.mxfp8_quantize_dim0(wn)
    ref, bound = OG.grouped_mm_fwd(OQ.dequant_mx(qa, sa), OQ.dequant_mx(qw, sw), offs)
    _check(out, ref, bound, "forward")
    # dgrad: dY along N, W along N (its dim 1)
    qdy, sdy = OQ.mxfp8_quantize_dim0(dyn)
    qwt, swt = OQ.mxfp8_quantize_dim1(wn)
    ref, bound = OG.grouped_mm_dgrad(OQ.dequant_mx(qdy, sdy), OQ.dequant_mx(qwt, swt), offs)
    _check(da, ref, bound, "dgrad")
    # wgrad: dY and A along the routed tokens (dim 1 of each)
    qdyt, sdyt = OQ.mxfp8_quantize_dim1(dyn)
    qat, sat = OQ.mxfp8_quantize_dim1(an)
    ref, bound = OG.grouped_mm_wgrad(OQ.dequant_mx(qdyt, sdyt), OQ.dequant_mx(qat, sat), offs)
    _check(dw, ref, bound, "wgrad")


def test_layer_equals_single_calls(F):
    sizes = [96, 0, 160, 32, 0, 256]
    offs = torch.from_numpy(W.offsets_from_sizes(sizes)).to(DEV)
    M, E, N, K = sum(sizes), len(sizes), 192, 256
    a, w, dy = _bf16((M, K), 81).to(DEV), _bf16((E, N, K), 82, 0.05).to(DEV), _bf16((M, N), 83).to(DEV)
    out, ws = F.fp8moe_mxfp8_moe_fwd(a, w, offs)
    da, dw = F.fp8moe_mxfp8_moe_bwd(dy, offs, ws, K)
    r_out, r_da, r_dw = _chain(F, a, w, dy, offs)
    assert torch.equal(out, r_out) and torch.equal(da, r_da) and torch.equal(dw, r_dw)
    # one backward result at a time: the other is not produced
    da1, dw1 = F.fp8moe_mxfp8_moe_bwd(dy, offs, ws, K, need_dw=False)
    assert dw1 is None and torch.equal(da1, r_da)
    da2, dw2 = F.fp8moe_mxfp8_moe_bwd(dy, offs, ws, K, need_da=False)
    assert da2 is None and torch.equal(dw2, r_dw)
    assert F.fp8moe_get_device_status() == 0


def test_layer_no_tokens(F):
    E, N, K = 3, 64, 96
    offs = torch.zeros(E, dtype=torch.int32, device=DEV)
    a = torch.zeros(0, K, dtype=torch.bfloat16, device=DEV)
    w = _bf16((E, N, K), 91).to(DEV)
    out, ws = F.fp8moe_mxfp8_moe_fwd(a, w, offs)
    dy = torch.zeros(0, N, dtype=torch.bfloat16, device=DEV)
    da, dw = F.fp8moe_mxfp8_moe_bwd(dy, offs, ws, K)
    assert out.shape == (0, N) and da.shape == (0, K)
    assert torch.count_nonzero(dw).item() == 0
    assert F.fp8moe_get_device_status() == 0


def test_layer_rejects_bad_sizes(F):
    a = torch.zeros(64, 48, dtype=torch.bfloat16, device=DEV)     # K % 32 != 0
    w = torch.zeros(2, 64, 48, dtype=torch.bfloat16, device=DEV)
    offs = torch.tensor([32, 64], dtype=torch.int32, device=DEV)
    with pytest.raises(F.Fp8MoeError):
        F.fp8moe_mxfp8_moe_fwd(a, w, offs)
    a = torch.zeros(64, 64, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(2, 64, 64, dtype=torch.bfloat16, device=DEV)
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(F.Fp8MoeError):
        F.fp8moe_mxfp8_moe_fwd(a, w, offs, workspace=small)


def test_layer_scout_size_equals_single_calls(F):
    """Llama4-Scout W1 layer: the composite against the single-call chain,
    bit for bit, on the seeded workload."""
    wl = W.get_workload("scout")
    offs = torch.from_numpy(wl.offs()).to(DEV)
    a = W.make_activations(wl, "A", device=DEV)
    w = W.make_weights(wl, "W1", device=DEV)
    dy = _bf16((a.shape[0], w.shape[1]), 95).to(DEV)
    out, ws = F.fp8moe_mxfp8_moe_fwd(a, w, offs)
    da, dw = F.fp8moe_mxfp8_moe_bwd(dy, offs, ws, w.shape[2])
    del ws
    r_out, r_da, r_dw = _chain(F, a, w, dy, offs)
    assert torch.equal(out, r_out) and torch.equal(da, r_da) and torch.equal(dw, r_dw)
    assert F.fp8moe_get_device_status() == 0
