"""GPU parity of the scaled grouped GEMM (forward / dgrad / wgrad) against the
CPU oracle.

The FP8 operands and their scales are produced by the *oracle* from the seeded
bf16 inputs and uploaded, so the GEMM is checked on its own; the expected
values are the oracle's float64 grouped GEMM of the dequantized operands.
Tolerance (elementwise): |gpu - ref| <= 8e-3 |ref| + 1e-3 sum_k |a_k b_k|.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats as OF, grouped_mm as OG, quant as OQ, swizzle as OS

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
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16).float().numpy()


def _d(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def check(out, ref, bound, what=""):
    got = out.float().cpu().numpy()
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    lim = RTOL * np.abs(ref) + BTOL * bound
    bad = err > lim
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst " \
                          f"{float((err - lim).max())} at {np.unravel_index(np.argmax(err - lim), err.shape)}"


# ----------------------------------------------------------------------------
# operand builders (oracle side)
# ----------------------------------------------------------------------------

def mx_fwd_case(a, w, offs):
    """a [M,K], w [E,N,K] (bf16 values) -> device operands + oracle reference."""
    qa, sa = OQ.mxfp8_quantize_dim0(a)
    qw, sw = OQ.mxfp8_quantize_dim0(w)
    ref, bound = OG.grouped_mm_fwd(OQ.dequant_mx(qa, sa), OQ.dequant_mx(qw, sw), offs)
    dev = (_d(qa), _d(OS.swizzle(sa, offs, OS.GROUP_ROWS)), _d(qw), _d(OS.swizzle(sw)))
    return dev, ref, bound


def mx_dgrad_case(dy, w, offs):
    """dy [M,N], w [E,N,K]: the weight is quantized along N (dim1) -> Wt [E,K,N]."""
    qdy, sdy = OQ.mxfp8_quantize_dim0(dy)
    qwt, swt = OQ.mxfp8_quantize_dim1(w)
    ref, bound = OG.grouped_mm_dgrad(OQ.dequant_mx(qdy, sdy), OQ.dequant_mx(qwt, swt), offs)
    dev = (_d(qdy), _d(OS.swizzle(sdy, offs, OS.GROUP_ROWS)), _d(qwt), _d(OS.swizzle(swt)))
    return dev, ref, bound


def mx_wgrad_case(dy, a, offs):
    """dY^T and A^T quantized along the token dim (dim1), column-grouped scales."""
    qdyt, sdyt = OQ.mxfp8_quantize_dim1(dy)
    qat, sat = OQ.mxfp8_quantize_dim1(a)
    ref, bound = OG.grouped_mm_wgrad(OQ.dequant_mx(qdyt, sdyt), OQ.dequant_mx(qat, sat), offs)
    dev = (_d(qdyt), _d(OS.swizzle(sdyt, offs, OS.GROUP_COLS)), _d(qat), _d(OS.swizzle(sat, offs, OS.GROUP_COLS)))
    return dev, ref, bound


def rw_fwd_case(a, w, offs):
    qa, ia = OQ.quantize_rowwise(a)
    E, N, K = w.shape
    qw, iw = OQ.quantize_rowwise(w.reshape(E * N, K))
    ref, bound = OG.grouped_mm_fwd(OQ.dequant_rows(qa, ia), OQ.dequant_rows(qw, iw).reshape(E, N, K), offs)
    return (_d(qa), _d(ia), _d(qw.reshape(E, N, K)), _d(iw.reshape(E, N))), ref, bound


def rw_dgrad_case(dy, w, offs):
    qdy, idy = OQ.quantize_rowwise(dy)
    qwt, iwt = OQ.quantize_colwise_3d(w, transpose_out=True)          # [E,K,N], scales [E,K]
    wt_deq = OF.decode(qwt) * iwt[:, :, None].astype(np.float64)
    ref, bound = OG.grouped_mm_dgrad(OQ.dequant_rows(qdy, idy), wt_deq, offs)
    return (_d(qdy), _d(idy), _d(qwt), _d(iwt)), ref, bound


def rw_wgrad_case(dy, a, offs):
    qdyt, idyt = OQ.quantize_colwise_jagged(dy, offs, transpose_out=True)   # [N, Mt], [E, N]
    qat, iat = OQ.quantize_colwise_jagged(a, offs, transpose_out=True)      # [K, Mt], [E, K]
    starts, ends = OQ.group_bounds(offs)
    P = OQ.padded_starts(offs, 32)
    E = len(offs)
    dyt_deq = np.zeros(qdyt.shape)
    at_deq = np.zeros(qat.shape)
    for e in range(E):
        g = ends[e] - starts[e]
        c = slice(P[e], P[e] + g)
        dyt_deq[:, c] = OF.decode(qdyt[:, c]) * idyt[e][:, None]
        at_deq[:, c] = OF.decode(qat[:, c]) * iat[e][:, None]
    ref, bound = OG.grouped_mm_wgrad(dyt_deq, at_deq, offs, col0=P)
    return (_d(qdyt), _d(idyt), _d(qat), _d(iat)), ref, bound


SHAPES = {
    # name: (group sizes, N, K)
    "tiny": (list(W.group_sizes("tiny")), 512, 256),
    "ragged": ([64, 0, 352, 32, 160], 320, 384),
    "dense": ([512], 1024, 512),
    "wide_k": ([128, 96, 0, 288], 256, 1408 + 128),
    # groups of 512 tokens or more on average: the wgrad stores 64-column
    # slices; 352 columns leave a half slice, 288 rows a partial tile
    "long_groups": ([704, 0, 896], 288, 352),
}
RW_SHAPES = {
    "tiny": (list(W.group_sizes("tiny")), 512, 256),
    "odd_groups": ([149, 0, 306, 7, 200], 1408 // 4, 2048 // 8),
    "dense": ([300], 272, 144),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_mx_fwd(F, name):
    sizes, N, K = SHAPES[name]
    offs = W.offsets_from_sizes(sizes)
    M = int(sum(sizes))
    a = _bf16((M, K), 11 + M)
    w = _bf16((len(sizes), N, K), 12 + N, 0.05)
    (qa, sa, qw, sw), ref, bound = mx_fwd_case(a, w, offs)
    out = F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, qa, sa, qw, sw, _d(offs))
    assert F.fp8moe_get_device_status() == 0
    check(out, ref, bound, f"mx fwd {name}")


@pytest.mark.parametrize("name", list(SHAPES))
def test_mx_dgrad(F, name):
    sizes, N, K = SHAPES[name]
    offs = W.offsets_from_sizes(sizes)
    M = int(sum(sizes))
    dy = _bf16((M, N), 21 + M)
    w = _bf16((len(sizes), N, K), 22 + N, 0.05)
    (qdy, sdy, qwt, swt), ref, bound = mx_dgrad_case(dy, w, offs)
    out = F.fp8moe_scaled_grouped_mm_dgrad(F.MXFP8, qdy, sdy, qwt, swt, _d(offs))
    assert F.fp8moe_get_device_status() == 0
    check(out, ref, bound, f"mx dgrad {name}")


@pytest.mark.parametrize("name", list(SHAPES))
def test_mx_wgrad(F, name):
    sizes, N, K = SHAPES[name]
    offs = W.offsets_from_sizes(sizes)
    M = int(sum(sizes))
    dy = _bf16((M, N), 31 + M)
    a = _bf16((M, K), 32 + K)
    (qdyt, sdyt, qat, sat), ref, bound = mx_wgrad_case(dy, a, offs)
    out = F.fp8moe_scaled_grouped_mm_wgrad(F.MXFP8, qdyt, sdyt, qat, sat, _d(offs), M)
    assert F.fp8moe_get_device_status() == 0
    check(out, ref, bound, f"mx wgrad {name}")
    for e, g in enumerate(sizes):
        if g == 0:
            assert torch.all(out[e] == 0)


@pytest.mark.parametrize("name", list(RW_SHAPES))
def test_rowwise_fwd(F, name):
    sizes, N, K = RW_SHAPES[name]
    offs = W.offsets_from_sizes(sizes)
    M = int(sum(sizes))
    a = _bf16((M, K), 41 + M)
    w = _bf16((len(sizes), N, K), 42 + N, 0.05)
    (qa, ia, qw, iw), ref, bound = rw_fwd_case(a, w, offs)
    out = F.fp8moe_scaled_grouped_mm_fwd(F.ROWWISE, qa, ia, qw, iw, _d(offs))
    assert F.fp8moe_get_device_status() == 0
    check(out, ref, bound, f"rowwise fwd {name}")


@pytest.mark.parametrize("name", list(RW_SHAPES))
def test_rowwise_dgrad(F, name):
    sizes, N, K = RW_SHAPES[name]
    offs = W.offsets_from_sizes(sizes)
    M = int(sum(sizes))
    dy = _bf16((M, N), 51 + M)
    w = _bf16((len(sizes), N, K), 52 + N, 0.05)
    (qdy, idy, qwt, iwt), ref, bound = rw_dgrad_case(dy, w, offs)
    out = F.fp8moe_scaled_grouped_mm_dgrad(F.ROWWISE, qdy, idy, qwt, iwt, _d(offs))
    assert F.fp8moe_get_device_status() == 0
    check(out, ref, bound, f"rowwise dgrad {name}")


@pytest.mark.parametrize("name", list(RW_SHAPES))
def test_rowwise_wgrad(F, name):
    sizes, N, K = RW_SHAPES[name]
    offs = W.offsets_from_sizes(sizes)
    M = int(sum(sizes))
    dy = _bf16((M, N), 61 + M)
    a = _bf16((M, K), 62 + K)
    (qdyt, idyt, qat, iat), ref, bound = rw_wgrad_case(dy, a, offs)
    out = F.fp8moe_scaled_grouped_mm_wgrad(F.ROWWISE, qdyt, idyt, qat, iat, _d(offs), M)
    assert F.fp8moe_get_device_status() == 0
    check(out, ref, bound, f"rowwise wgrad {name}")


def test_bad_offsets_set_status(F):
    sizes, N, K = SHAPES["tiny"]
    offs = W.offsets_from_sizes(sizes)
    M = int(sum(sizes))
    a = _bf16((M, K), 71)
    w = _bf16((len(sizes), N, K), 72, 0.05)
    (qa, sa, qw, sw), _, _ = mx_fwd_case(a, w, offs)
    bad = torch.tensor([96, 64, 96, 1024], dtype=torch.int32, device=DEV)     # decreasing
    F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, qa, sa, qw, sw, bad)
    assert F.fp8moe_get_device_status() == 5
    bad = torch.tensor([96, 96, 100, 1024], dtype=torch.int32, device=DEV)    # not a multiple of 32
    F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, qa, sa, qw, sw, bad)
    assert F.fp8moe_get_device_status() == 5
    assert F.fp8moe_get_device_status() == 0


@pytest.mark.parametrize("E", [600, 1024])
def test_many_groups_fwd(F, E):
    """More groups than the 512-entry tables of the default variant: the
    launch takes the variant with 1024-entry tables (a 5-deep ring, the same
    cta_group::2 pairs); many groups are empty."""
    rng = np.random.default_rng(5 + E)
    sizes = (rng.integers(0, 3, size=E) * 32).tolist()
    offs = W.offsets_from_sizes(sizes)
    M, N, K = int(sum(sizes)), 256, 128
    a = _bf16((M, K), 81)
    w = _bf16((len(sizes), N, K), 82, 0.05)
    (qa, sa, qw, sw), ref, bound = mx_fwd_case(a, w, offs)
    out = F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, qa, sa, qw, sw, _d(offs))
    assert F.fp8moe_get_device_status() == 0
    check(out, ref, bound, f"mx fwd, {E} groups")


def test_many_groups_rowwise_fwd(F):
    """The rowwise recipe with E = 1024 groups of odd sizes (many empty)."""
    rng = np.random.default_rng(17)
    sizes = rng.integers(0, 40, size=1024)
    sizes[rng.random(1024) < 0.3] = 0
    sizes = sizes.tolist()
    offs = W.offsets_from_sizes(sizes)
    M, N, K = int(sum(sizes)), 272, 144
    a = _bf16((M, K), 83)
    w = _bf16((len(sizes), N, K), 84, 0.05)
    (qa, ia, qw, iw), ref, bound = rw_fwd_case(a, w, offs)
    out = F.fp8moe_scaled_grouped_mm_fwd(F.ROWWISE, qa, ia, qw, iw, _d(offs))
    assert F.fp8moe_get_device_status() == 0
    check(out, ref, bound, "rowwise fwd, 1024 groups")


def test_many_groups_wgrad(F):
    """MXFP8 wgrad with 1024 groups (most empty, checked to be exactly 0)."""
    rng = np.random.default_rng(23)
    sizes = (rng.integers(0, 2, size=1024) * rng.integers(1, 3, size=1024) * 32).tolist()
    offs = W.offsets_from_sizes(sizes)
    M, N, K = int(sum(sizes)), 128, 256
    dy = _bf16((M, N), 85)
    a = _bf16((M, K), 86)
    (qdyt, sdyt, qat, sat), ref, bound = mx_wgrad_case(dy, a, offs)
    out = F.fp8moe_scaled_grouped_mm_wgrad(F.MXFP8, qdyt, sdyt, qat, sat, _d(offs), M)
    assert F.fp8moe_get_device_status() == 0
    check(out, ref, bound, "mx wgrad, 1024 groups")


def test_pipeline_wait_timeout_sets_status(F):
    """Fault injection without a GPU fault: the one-shot testing hook makes
    the first pair of the next launch keep its first accumulator, so the
    epilogue's bounded wait (2 s) runs out.  The kernel reports
    FP8MOE_ERR_TIMEOUT; every CTA waits for its own copies and MMAs before
    releasing TMEM, so the context stays usable and the next GEMM (the hook
    is spent) is exact again."""
    offs = W.offsets_from_sizes([64, 0, 352, 32, 160])
    a = _bf16((608, 256), 91)
    w = _bf16((5, 512, 256), 92, 0.05)
    (qa, sa, qw, sw), ref, bound = mx_fwd_case(a, w, offs)
    d_offs = _d(offs)
    F.fp8moe_testing_stall_next_gemm()
    F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, qa, sa, qw, sw, d_offs)
    assert F.fp8moe_get_device_status() == 6          # FP8MOE_ERR_TIMEOUT
    out = F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, qa, sa, qw, sw, d_offs)
    assert F.fp8moe_get_device_status() == 0
    check(out, ref, bound, "fwd after a timed-out launch")


def test_status_taken_on_another_stream(F):
    """An offsets error set by a launch on one stream is read (and cleared)
    through a status call on another stream once that stream has waited."""
    sizes, N, K = SHAPES["tiny"]
    offs = W.offsets_from_sizes(sizes)
    M = int(sum(sizes))
    a = _bf16((M, K), 93)
    w = _bf16((len(sizes), N, K), 94, 0.05)
    (qa, sa, qw, sw), _, _ = mx_fwd_case(a, w, offs)
    bad = torch.tensor([96, 64, 96, 1024], dtype=torch.int32, device=DEV)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, qa, sa, qw, sw, bad, stream=s1)
    s2.wait_stream(s1)
    assert F.fp8moe_get_device_status(stream=s2) == 5
    assert F.fp8moe_get_device_status(stream=s2) == 0
