"""GPU parity of blockwise FP8 (one fp32 scale per 1 x 128, 128 x 128 or
per-group 128-token tile) against the CPU oracle: the three quantizations
bit-exact (codes and scales), and the blockwise grouped GEMMs (forward,
dgrad, wgrad) within the grouped GEMM tolerance
|gpu - ref| <= 8e-3 |ref| + 1e-3 sum_k |a_k b_k|, both on operands the
oracle quantized (the GEMM alone) and end to end through the GPU
quantization."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import blockwise as BW, formats as OF, grouped_mm as OG

pytestmark = pytest.mark.gpu
DEV = "cuda"
RTOL, BTOL = 8e-3, 1e-3
KINDS = [(0, OF.FN), (1, OF.FNUZ)]


@pytest.fixture(scope="module")
def F():
    from mxfp8_moe_quantization_gb300 import build as B
    B.build()
    import mxfp8_moe_quantization_gb300 as m
    return m


def _bf16(shape, seed, scale=1.0, spread=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(*shape, generator=g) * scale
    if spread:   # rows of very different magnitude, so tiles get different scales
        x = x * torch.exp(torch.empty(*shape[:-1], 1).uniform_(-3, 3, generator=g))
    return x.to(torch.bfloat16)


def _np(t):
    return t.float().cpu().numpy()


def _d(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _check(out, ref, bound, what):
    got = _np(out)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    lim = RTOL * np.abs(ref) + BTOL * bound
    assert np.all(err <= lim), f"{what}: {int((err > lim).sum())} outside; worst excess {float((err - lim).max())}"


# ----------------------------------------------------------------------------
# quantization
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("kind,okind", KINDS)
@pytest.mark.parametrize("R,C", [(1, 128), (37, 384), (1000, 1280), (16, 5120)])
def test_rows_parity(F, kind, okind, R, C):
    x = _bf16((R, C), R + C)
    if R > 3:
        x[3, :128] = 0.0
    q, inv = F.fp8moe_quantize_blockwise_rows(x.to(DEV), kind)
    rq, rinv = BW.quantize_blockwise_rows(_np(x), okind)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(inv.cpu().numpy(), rinv)


@pytest.mark.parametrize("kind,okind", KINDS)
@pytest.mark.parametrize("E,N,K", [(1, 128, 128), (3, 256, 384), (2, 640, 256)])
def test_weight_parity(F, kind, okind, E, N, K):
    w = _bf16((E, N, K), E * N + K, 0.02)
    w[0, :128, :128] = 0.0                                   # an all-zero tile
    q, qt, inv = F.fp8moe_quantize_blockwise_weight(w.to(DEV), kind)
    rq, rinv = BW.quantize_blockwise_weight(_np(w), okind)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(qt.cpu().numpy(), np.ascontiguousarray(rq.transpose(0, 2, 1)))
    assert np.array_equal(inv.cpu().numpy(), rinv)
    # one direction alone
    q1, qt1, _ = F.fp8moe_quantize_blockwise_weight(w.to(DEV), kind, transposed=False)
    _, qt2, _ = F.fp8moe_quantize_blockwise_weight(w.to(DEV), kind, plain=False)
    assert qt1 is None and torch.equal(q1, q) and torch.equal(qt2, qt)


@pytest.mark.parametrize("kind,okind", KINDS)
@pytest.mark.parametrize("sizes,C", [([96, 0, 320, 32, 0, 160], 48), ([0, 0, 64], 256), ([4096], 144),
                                     ([32] * 9, 16),
                                     # from 128 columns on, the TMA-ring kernel: enough units
                                     # (81 token blocks x 16 column tiles) for every CTA's
                                     # six-slot ring to wrap, blocks ending inside groups
                                     ([3008, 0, 4992, 2016, 96], 2048)])
def test_tokens_parity(F, kind, okind, sizes, C):
    offs = W.offsets_from_sizes(sizes)
    M = int(sum(sizes))
    x = _bf16((M, C), M + C)
    qt, inv = F.fp8moe_quantize_blockwise_tokens(x.to(DEV), _d(offs), kind)
    assert F.fp8moe_get_device_status() == 0
    rq, rinv = BW.quantize_blockwise_tokens(_np(x), offs, okind)
    assert np.array_equal(qt.cpu().numpy(), rq)
    nb = len(rinv)
    assert np.array_equal(inv.cpu().numpy()[:nb], rinv)


def test_tokens_bad_offsets(F):
    x = torch.zeros(128, 32, dtype=torch.bfloat16, device=DEV)
    for bad in ([64, 48], [100, 128], [64, 96]):        # decreasing, not a multiple of 32, short
        F.fp8moe_quantize_blockwise_tokens(x, torch.tensor(bad, dtype=torch.int32, device=DEV))
        assert F.fp8moe_get_device_status() == 5
    assert F.fp8moe_get_device_status() == 0


# ----------------------------------------------------------------------------
# grouped GEMM
# ----------------------------------------------------------------------------

def _oracle_operands(a, w, dy, offs):
    qa, sa = BW.quantize_blockwise_rows(a)
    qw, sw = BW.quantize_blockwise_weight(w)
    qdy, sdy = BW.quantize_blockwise_rows(dy)
    qdyt, sdyt = BW.quantize_blockwise_tokens(dy, offs)
    qat, sat = BW.quantize_blockwise_tokens(a, offs)
    return qa, sa, qw, sw, qdy, sdy, qdyt, sdyt, qat, sat


def _refs(ops, offs):
    qa, sa, qw, sw, qdy, sdy, qdyt, sdyt, qat, sat = ops
    wd = BW.dequant_weight(qw, sw)
    fwd = OG.grouped_mm_fwd(BW.dequant_rows(qa, sa), wd, offs)
    dgrad = OG.grouped_mm_dgrad(BW.dequant_rows(qdy, sdy), wd.transpose(0, 2, 1), offs)
    wgrad = OG.grouped_mm_wgrad(BW.dequant_tokens(qdyt, sdyt, offs), BW.dequant_tokens(qat, sat, offs), offs)
    return fwd, dgrad, wgrad


def _pad_blocks(F, s, M, E):
    """Token-tile scales in a buffer of the size the GPU quantization uses."""
    out = np.zeros((F.fp8moe_blockwise_token_blocks(M, E), s.shape[1]), np.float32)
    out[:len(s)] = s
    return out


@pytest.mark.parametrize("sizes,N,K", [([96, 0, 352, 32, 160], 256, 384), ([0, 128, 0], 384, 128),
                                       ([544, 64, 32, 0, 416], 640, 256)])
def test_gemm_on_oracle_operands(F, sizes, N, K):
    offs = W.offsets_from_sizes(sizes)
    M, E = int(sum(sizes)), len(sizes)
    a, w, dy = _np(_bf16((M, K), 31)), _np(_bf16((E, N, K), 32, 0.05)), _np(_bf16((M, N), 33))
    ops = _oracle_operands(a, w, dy, offs)
    (rf, bf), (rd, bd), (rw, bw) = _refs(ops, offs)
    qa, sa, qw, sw, qdy, sdy, qdyt, sdyt, qat, sat = ops
    d_offs = _d(offs)
    out = F.fp8moe_scaled_grouped_mm_fwd(F.BLOCKWISE, _d(qa), _d(sa), _d(qw), _d(sw), d_offs)
    _check(out, rf, bf, "blockwise forward")
    qwt = np.ascontiguousarray(qw.transpose(0, 2, 1))
    da = F.fp8moe_scaled_grouped_mm_dgrad(F.BLOCKWISE, _d(qdy), _d(sdy), _d(qwt), _d(sw), d_offs)
    _check(da, rd, bd, "blockwise dgrad")
    dw = F.fp8moe_scaled_grouped_mm_wgrad(F.BLOCKWISE, _d(qdyt), _d(_pad_blocks(F, sdyt, M, E)), _d(qat),
                                          _d(_pad_blocks(F, sat, M, E)), d_offs, M)
    _check(dw, rw, bw, "blockwise wgrad")
    assert F.fp8moe_get_device_status() == 0


def test_gemm_end_to_end_through_gpu_quantization(F):
    """Routed-layer shapes (8 experts, 32-padded Dirichlet groups): every
    operand quantized on the GPU, every GEMM against the oracle chain."""
    rng = np.random.default_rng(7)
    sizes = list(rng.multinomial(64, rng.dirichlet(np.ones(8))) * 32)
    sizes[3] = 0
    offs = W.offsets_from_sizes(sizes)
    M, E, N, K = int(sum(sizes)), 8, 1024, 768
    a, w, dy = _bf16((M, K), 41), _bf16((E, N, K), 42, 0.05), _bf16((M, N), 43)
    d_offs = _d(offs)
    qa, sa = F.fp8moe_quantize_blockwise_rows(a.to(DEV))
    qw, qwt, sw = F.fp8moe_quantize_blockwise_weight(w.to(DEV))
    qdy, sdy = F.fp8moe_quantize_blockwise_rows(dy.to(DEV))
    qdyt, sdyt = F.fp8moe_quantize_blockwise_tokens(dy.to(DEV), d_offs)
    qat, sat = F.fp8moe_quantize_blockwise_tokens(a.to(DEV), d_offs)
    out = F.fp8moe_scaled_grouped_mm_fwd(F.BLOCKWISE, qa, sa, qw, sw, d_offs)
    da = F.fp8moe_scaled_grouped_mm_dgrad(F.BLOCKWISE, qdy, sdy, qwt, sw, d_offs)
    dw = F.fp8moe_scaled_grouped_mm_wgrad(F.BLOCKWISE, qdyt, sdyt, qat, sat, d_offs, M)
    assert F.fp8moe_get_device_status() == 0
    (rf, bf), (rd, bd), (rw, bw) = _refs(_oracle_operands(_np(a), _np(w), _np(dy), offs), offs)
    _check(out, rf, bf, "forward")
    _check(da, rd, bd, "dgrad")
    _check(dw, rw, bw, "wgrad")


def test_gemm_rejects_unaligned_sizes(F):
    z = torch.zeros(64, 192, dtype=torch.uint8, device=DEV)
    s = torch.zeros(2, 64, dtype=torch.float32, device=DEV)
    wq = torch.zeros(1, 128, 192, dtype=torch.uint8, device=DEV)
    offs = torch.tensor([64], dtype=torch.int32, device=DEV)
    with pytest.raises(F.Fp8MoeError):       # K = 192 is not a multiple of 128
        F.fp8moe_scaled_grouped_mm_fwd(F.BLOCKWISE, z, s, wq, s, offs)
