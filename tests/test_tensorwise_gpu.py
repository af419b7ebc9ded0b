"""GPU parity of tensorwise FP8 (one scale per tensor) against the CPU oracle:
quantization in every output layout (bit-exact codes and scale) and the
grouped GEMMs with the tensorwise recipe (within the GEMM tolerance)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats as OF, grouped_mm as OG, quant as OQ

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


def _kind(F, k):
    return F.E4M3FN if k == OF.FN else F.E4M3FNUZ


@pytest.mark.parametrize("kind", [OF.FN, OF.FNUZ])
@pytest.mark.parametrize("shape", [(1024, 256), (7, 9), (3, 96, 160), (1, 5000, 48), (1023, 4099), (4096, 2048)])
def test_tensorwise_plain(F, kind, shape):
    x = _bf16(shape, sum(shape) + 3, 2.0)
    q, inv = F.fp8moe_quantize_tensorwise(x.to(DEV), kind=_kind(F, kind))
    rq, rinv = OQ.quantize_tensorwise(_np(x), kind)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert inv.cpu().numpy()[0] == rinv
    assert F.fp8moe_get_device_status() == 0


@pytest.mark.parametrize("kind", [OF.FN, OF.FNUZ])
def test_tensorwise_dense_transposed(F, kind):
    x = _bf16((4, 160, 96), 21, 0.05)
    x[2, 17, 33] = 3.0                                   # one outlier sets the scale
    q, inv = F.fp8moe_quantize_tensorwise(x.to(DEV), transpose_out=True, kind=_kind(F, kind))
    rq, rinv = OQ.quantize_tensorwise(_np(x), kind)
    assert np.array_equal(q.cpu().numpy(), np.ascontiguousarray(rq.transpose(0, 2, 1)))
    assert inv.cpu().numpy()[0] == rinv


@pytest.mark.parametrize("sizes", [[96, 0, 170, 33, 0], [0, 0, 64], [5]])
def test_tensorwise_jagged_transposed(F, sizes):
    M = int(sum(sizes))
    x = _bf16((M, 48), M + 5, 1.0)
    offs = W.offsets_from_sizes(sizes)
    q, inv = F.fp8moe_quantize_tensorwise(x.to(DEV), torch.from_numpy(offs).to(DEV), transpose_out=True)
    rq, rinv = OQ.quantize_tensorwise(_np(x), OF.FN)
    starts, ends = OQ.group_bounds(offs)
    P = OQ.padded_starts(offs, 32)
    ref = np.zeros((48, F.fp8moe_jagged_t_cols(M, len(sizes))), np.uint8)
    for e in range(len(sizes)):
        ref[:, P[e]:P[e] + ends[e] - starts[e]] = rq[starts[e]:ends[e]].T
    assert np.array_equal(q.cpu().numpy(), ref)
    assert inv.cpu().numpy()[0] == rinv
    assert F.fp8moe_get_device_status() == 0


def test_tensorwise_zero_and_empty(F):
    z = torch.zeros(64, 32, dtype=torch.bfloat16, device=DEV)
    q, inv = F.fp8moe_quantize_tensorwise(z)
    rq, rinv = OQ.quantize_tensorwise(np.zeros((64, 32), np.float32), OF.FN)
    assert np.array_equal(q.cpu().numpy(), rq) and inv.cpu().numpy()[0] == rinv
    e = torch.zeros(0, 32, dtype=torch.bfloat16, device=DEV)
    _, inv0 = F.fp8moe_quantize_tensorwise(e, kind=F.E4M3FNUZ)
    assert inv0.cpu().numpy()[0] == OQ.quantize_tensorwise(np.zeros((0, 32), np.float32), OF.FNUZ)[1]


def _check(out, ref, bound, what):
    got = out.float().cpu().numpy()
    err = np.abs(got - ref)
    lim = RTOL * np.abs(ref) + BTOL * bound
    assert np.all(err <= lim), f"{what}: worst excess {float((err - lim).max())}"


def _deq(q, inv):
    return OF.decode(q) * np.float64(inv)


@pytest.mark.parametrize("sizes,N,K", [([64, 0, 352, 32, 160], 320, 384), ([149, 0, 306, 7, 200], 352, 256)])
def test_tensorwise_gemms(F, sizes, N, K):
    offs = W.offsets_from_sizes(sizes)
    M, E = int(sum(sizes)), len(sizes)
    d_offs = torch.from_numpy(offs).to(DEV)
    a = _bf16((M, K), 61, 1.0)
    w = _bf16((E, N, K), 62, 0.05)
    dy = _bf16((M, N), 63, 1.0)
    # forward: A [M, K], W [E, N, K]
    qa, sa = F.fp8moe_quantize_tensorwise(a.to(DEV))
    qw, sw = F.fp8moe_quantize_tensorwise(w.to(DEV))
    out = F.fp8moe_scaled_grouped_mm_fwd(F.TENSORWISE, qa, sa, qw, sw, d_offs)
    ra, rsa = OQ.quantize_tensorwise(_np(a), OF.FN)
    rw, rsw = OQ.quantize_tensorwise(_np(w), OF.FN)
    ref, bound = OG.grouped_mm_fwd(_deq(ra, rsa), _deq(rw, rsw), offs)
    _check(out, ref, bound, "tensorwise fwd")
    # dgrad: dY [M, N], W^T [E, K, N]
    qdy, sdy = F.fp8moe_quantize_tensorwise(dy.to(DEV))
    qwt, swt = F.fp8moe_quantize_tensorwise(w.to(DEV), transpose_out=True)
    da = F.fp8moe_scaled_grouped_mm_dgrad(F.TENSORWISE, qdy, sdy, qwt, swt, d_offs)
    rdy, rsdy = OQ.quantize_tensorwise(_np(dy), OF.FN)
    ref, bound = OG.grouped_mm_dgrad(_deq(rdy, rsdy), _deq(rw, rsw).transpose(0, 2, 1), offs)
    _check(da, ref, bound, "tensorwise dgrad")
    # wgrad: dY^T, A^T in the group-padded transposed layout
    qdyt, sdyt = F.fp8moe_quantize_tensorwise(dy.to(DEV), d_offs, transpose_out=True)
    qat, sat = F.fp8moe_quantize_tensorwise(a.to(DEV), d_offs, transpose_out=True)
    dw = F.fp8moe_scaled_grouped_mm_wgrad(F.TENSORWISE, qdyt, sdyt, qat, sat, d_offs, M)
    P = OQ.padded_starts(offs, 32)
    starts, ends = OQ.group_bounds(offs)
    Mt = F.fp8moe_jagged_t_cols(M, E)
    dyt = np.zeros((N, Mt))
    at = np.zeros((K, Mt))
    for e in range(E):
        dyt[:, P[e]:P[e] + ends[e] - starts[e]] = _deq(rdy, rsdy)[starts[e]:ends[e]].T
        at[:, P[e]:P[e] + ends[e] - starts[e]] = _deq(ra, rsa)[starts[e]:ends[e]].T
    ref, bound = OG.grouped_mm_wgrad(dyt, at, offs, col0=P)
    _check(dw, ref, bound, "tensorwise wgrad")
    assert F.fp8moe_get_device_status() == 0


@pytest.mark.parametrize("which", ["A", "W1"])
def test_tensorwise_llama3_fullsize(F, which):
    """The bench's tensorwise workloads at full size (Llama3-8B X [8192,
    4096] and W [14336, 4096], plain layout: the one-launch streaming
    kernel with its grid-wide meeting), every code and the scale against the
    oracle."""
    wl = W.get_workload("llama3_8b")
    t = (W.make_activations(wl, "A", device=DEV) if which == "A"
         else W.make_weights(wl, "W1", device=DEV).reshape(wl.N, wl.K))
    q, inv = F.fp8moe_quantize_tensorwise(t)
    torch.cuda.synchronize()
    assert F.fp8moe_get_device_status() == 0
    rq, rinv = OQ.quantize_tensorwise(_np(t), OF.FN)
    assert inv.cpu().numpy()[0] == rinv
    assert np.array_equal(q.cpu().numpy(), rq)


def test_tensorwise_meeting_timeout_sets_status(F):
    """Fault injection without a GPU fault: the one-shot testing hook makes
    the first CTA of the next one-launch tensorwise kernel skip counting
    itself in at the grid-wide meeting, so every CTA's bounded wait (2 s)
    runs out; the launch reports FP8MOE_ERR_TIMEOUT, every CTA still waits for
    its own loads and releases its tensor memory, and the next call (the
    hook is spent) is exact again."""
    x = _bf16((2048, 1024), 77, 1.5)
    F.fp8moe_testing_stall_next_tensorwise()
    F.fp8moe_quantize_tensorwise(x.to(DEV))
    assert F.fp8moe_get_device_status() == 6          # FP8MOE_ERR_TIMEOUT
    q, inv = F.fp8moe_quantize_tensorwise(x.to(DEV))
    assert F.fp8moe_get_device_status() == 0
    rq, rinv = OQ.quantize_tensorwise(_np(x), OF.FN)
    assert np.array_equal(q.cpu().numpy(), rq) and inv.cpu().numpy()[0] == rinv
