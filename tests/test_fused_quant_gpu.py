"""GPU parity of the MXFP8 grouped GEMM whose prologue quantizes the bf16
activation (forward: A; dgrad: dY) inside the kernel.

Three checks per case, all on seeded inputs:
* the kernel's copy of the codes and e8m0 scales it fed the tensor cores
  equals the oracle's dim0 MXFP8 quantization of the bf16 operand, bit for
  bit (oracle/quant.py mxfp8_quantize_dim0);
* the output equals, bit for bit, the library's unfused chain (dim0
  quantization, GROUP_ROWS swizzle, MXFP8 grouped GEMM) on the same inputs;
* the output is within |gpu - ref| <= 8e-3 |ref| + 1e-3 sum_k |a_k b_k| of
  the oracle's float64 grouped GEMM of the dequantized operands.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import grouped_mm as OG, quant as OQ, swizzle as OS

pytestmark = pytest.mark.gpu
DEV = "cuda"
RTOL, BTOL = 8e-3, 1e-3


@pytest.fixture(scope="module")
def F():
    from mxfp8_moe_quantization_gb300 import build as B
    B.build()
    import mxfp8_moe_quantization_gb300 as m
    return m


def _bf16(shape, seed, scale=1.0, outliers=0.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(*shape, generator=g) * scale
    if outliers:
        m = torch.rand(*shape, generator=g) < outliers
        x = torch.where(m, x * 60.0, x)
    return x.to(torch.bfloat16)


def _d(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def _check(out, ref, bound, what):
    got = out.float().cpu().numpy()
    err = np.abs(got - ref)
    lim = RTOL * np.abs(ref) + BTOL * bound
    assert np.all(err <= lim), f"{what}: worst excess {float((err - lim).max())}"


CASES = {
    # name: (group sizes, N, K)
    "tiny": (list(W.group_sizes("tiny")), 512, 256),
    "ragged": ([64, 0, 352, 32, 160], 320, 384),
    "k_tail": ([96, 224, 0, 32], 256, 416),          # K = 3*128 + 32: a partial last k-stage
    "wide": ([512, 160], 768, 1536),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fwd_quant_a(F, name):
    sizes, N, K = CASES[name]
    offs = W.offsets_from_sizes(sizes)
    M, E = int(sum(sizes)), len(sizes)
    a = _bf16((M, K), 301 + M, outliers=0.003)
    w = _bf16((E, N, K), 302 + N, 0.05)
    af, wf = a.float().numpy(), w.float().numpy()
    rq, rs = OQ.mxfp8_quantize_dim0(af)
    qw, sw = OQ.mxfp8_quantize_dim0(wf)
    d_offs, d_qw, d_sw = _d(offs), _d(qw), _d(OS.swizzle(sw))
    out, a_q, a_s = F.fp8moe_mxfp8_grouped_mm_fwd_quant_a(a.to(DEV), d_qw, d_sw, d_offs, keep_quantized=True)
    assert F.fp8moe_get_device_status() == 0
    assert np.array_equal(a_q.cpu().numpy(), rq)
    assert np.array_equal(a_s.cpu().numpy(), rs)
    # the unfused chain of library calls
    q0, s0 = F.fp8moe_mxfp8_quantize_dim0(a.to(DEV))
    s0w = F.fp8moe_swizzle_scales_128x4(s0, d_offs, F.GROUP_ROWS)
    ref_chain = F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, q0, s0w, d_qw, d_sw, d_offs)
    assert torch.equal(out.view(torch.int16), ref_chain.view(torch.int16))
    ref, bound = OG.grouped_mm_fwd(OQ.dequant_mx(rq, rs), OQ.dequant_mx(qw, sw), offs)
    _check(out, ref, bound, f"fused fwd {name}")
    # without the optional copy
    out2 = F.fp8moe_mxfp8_grouped_mm_fwd_quant_a(a.to(DEV), d_qw, d_sw, d_offs)
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16))


@pytest.mark.parametrize("name", list(CASES))
def test_dgrad_quant_a(F, name):
    sizes, N, K = CASES[name]
    offs = W.offsets_from_sizes(sizes)
    M, E = int(sum(sizes)), len(sizes)
    dy = _bf16((M, N), 311 + M)
    w = _bf16((E, N, K), 312 + K, 0.05)
    dyf, wf = dy.float().numpy(), w.float().numpy()
    rq, rs = OQ.mxfp8_quantize_dim0(dyf)
    qwt, swt = OQ.mxfp8_quantize_dim1(wf)                      # [E, K, N], scales over N
    d_offs, d_qwt, d_swt = _d(offs), _d(qwt), _d(OS.swizzle(swt))
    out, q, s = F.fp8moe_mxfp8_grouped_mm_dgrad_quant_a(dy.to(DEV), d_qwt, d_swt, d_offs, keep_quantized=True)
    assert F.fp8moe_get_device_status() == 0
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy(), rs)
    q0, s0 = F.fp8moe_mxfp8_quantize_dim0(dy.to(DEV))
    s0w = F.fp8moe_swizzle_scales_128x4(s0, d_offs, F.GROUP_ROWS)
    ref_chain = F.fp8moe_scaled_grouped_mm_dgrad(F.MXFP8, q0, s0w, d_qwt, d_swt, d_offs)
    assert torch.equal(out.view(torch.int16), ref_chain.view(torch.int16))
    ref, bound = OG.grouped_mm_dgrad(OQ.dequant_mx(rq, rs), OQ.dequant_mx(qwt, swt), offs)
    _check(out, ref, bound, f"fused dgrad {name}")


def test_fwd_quant_a_many_groups(F):
    """600 groups (the variant with 1024-entry group tables), many empty,
    with special values in A: zeros, a block of bf16 subnormals, +-0."""
    rng = np.random.default_rng(41)
    sizes = (rng.integers(0, 3, size=600) * 32).tolist()
    offs = W.offsets_from_sizes(sizes)
    M, E, N, K = int(sum(sizes)), 600, 256, 128
    a = _bf16((M, K), 321)
    a[:, :32] = 0
    a[5, 32:64] = torch.tensor([1e-40] * 32).to(torch.bfloat16)
    a[7, 64:96] = -0.0
    w = _bf16((E, N, K), 322, 0.05)
    rq, rs = OQ.mxfp8_quantize_dim0(a.float().numpy())
    qw, sw = OQ.mxfp8_quantize_dim0(w.float().numpy())
    out, a_q, a_s = F.fp8moe_mxfp8_grouped_mm_fwd_quant_a(a.to(DEV), _d(qw), _d(OS.swizzle(sw)), _d(offs),
                                                          keep_quantized=True)
    assert F.fp8moe_get_device_status() == 0
    assert np.array_equal(a_q.cpu().numpy(), rq) and np.array_equal(a_s.cpu().numpy(), rs)
    ref, bound = OG.grouped_mm_fwd(OQ.dequant_mx(rq, rs), OQ.dequant_mx(qw, sw), offs)
    _check(out, ref, bound, "fused fwd, 600 groups")


def test_quant_a_host_errors(F):
    lib = F.lib()
    import ctypes
    p = ctypes.c_void_p(1 << 20)
    # contracting dimension not a multiple of 32; codes without scales
    assert lib.fp8moe_mxfp8_grouped_mm_fwd_quant_a(p, p, p, p, 4, 128, 256, 48, p, None, None, None) == 2
    assert lib.fp8moe_mxfp8_grouped_mm_dgrad_quant_a(p, p, p, p, 4, 128, 48, 256, p, None, None, None) == 2
    assert lib.fp8moe_mxfp8_grouped_mm_fwd_quant_a(p, p, p, p, 4, 128, 256, 256, p, p, None, None) == 1
