"""GPU parity of the quantization and swizzle kernels against the CPU oracle.

Codes and scales must match bit for bit.  Calls go through the C ABI (via the
thin binding).  Inputs come from the seeded generators in ``workloads`` or are
built here from e4m3 tie points.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats as OF, quant as OQ, swizzle as OS

pytestmark = pytest.mark.gpu

KINDS = [(0, OF.FN), (1, OF.FNUZ)]


@pytest.fixture(scope="module")
def F():
    from mxfp8_moe_quantization_gb300 import build as B
    B.build()
    import mxfp8_moe_quantization_gb300 as m
    torch.cuda.init()
    return m


DEV = "cuda"


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


def _np(t):
    return t.float().cpu().numpy()


def _tie_rows(R, C, seed, kind=OF.FN):
    """Rows whose scale is a power of two and whose elements sit on e4m3
    rounding midpoints, plus -0 and zeros."""
    rng = np.random.default_rng(seed)
    tab = OF.decode_table(kind)
    fin = np.sort(tab[np.isfinite(tab) & (tab >= 0)])
    mids = (fin[:-1] + fin[1:]) / 2
    cand = np.concatenate([fin, mids, [0.0]])
    vmax = OF.FP8_MAX[kind]
    x = np.empty((R, C))
    for r in range(R):
        j = int(rng.integers(-20, 20))
        row = rng.choice(cand, size=C) * rng.choice([-1.0, 1.0], size=C)
        row[int(rng.integers(0, C))] = vmax * (1 if r % 2 else -1)
        x[r] = row * 2.0 ** j
    x[0, 1] = -0.0
    t = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(t.float().numpy(), x.astype(np.float32)), "tie rows must be bf16-exact"
    return t


# ----------------------------------------------------------------------------
# rowwise
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("kind,okind", KINDS)
@pytest.mark.parametrize("R,C", [(1024, 256), (1024, 512), (37, 16), (5, 4096), (3, 14336), (2, 32768),
                                 (129, 1408), (64, 2048)])
def test_rowwise_parity(F, kind, okind, R, C):
    x = _bf16((R, C), R * 7 + C, 3.0)
    x[min(2, R - 1)] = 0.0
    q, inv = F.fp8moe_quantize_rowwise(x.to(DEV), kind)
    rq, rinv = OQ.quantize_rowwise(_np(x), okind)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(inv.cpu().numpy(), rinv)


@pytest.mark.parametrize("kind,okind", KINDS)
def test_rowwise_tie_points_and_stride(F, kind, okind):
    x = _tie_rows(64, 256, 5, okind)
    big = torch.zeros(64, 320, dtype=torch.bfloat16)
    big[:, :256] = x
    xv = big.to(DEV)[:, :256]                     # row stride 320 != C
    q, inv = F.fp8moe_quantize_rowwise(xv, kind)
    rq, rinv = OQ.quantize_rowwise(_np(x), okind)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(inv.cpu().numpy(), rinv)


def test_rowwise_tiny_workload(F):
    wl = W.get_workload("tiny")
    for which in ["A", "dY"]:
        x = W.make_activations(wl, which)
        for kind, okind in KINDS:
            q, inv = F.fp8moe_quantize_rowwise(x.to(DEV), kind)
            rq, rinv = OQ.quantize_rowwise(_np(x), okind)
            assert np.array_equal(q.cpu().numpy(), rq) and np.array_equal(inv.cpu().numpy(), rinv)


# ----------------------------------------------------------------------------
# colwise (dense 3D and jagged)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("kind,okind", KINDS)
@pytest.mark.parametrize("E,R,C", [(4, 256, 512), (2, 48, 32), (3, 64, 48), (1, 4096, 64),
                                   (1, 14336, 32), (1, 24576, 16),
                                   # transposed dense output runs one pass over clusters of 1-8
                                   # CTAs: 2-CTA slices of 704 rows with a partial 64-column tile,
                                   # 4-CTA slices with a ragged last one, 8-CTA slices of 800 rows
                                   # (two pieces each, the second 32 rows)
                                   (3, 1408, 80), (2, 2000, 48), (5, 6160, 16),
                                   # 8-CTA slices of 1504 rows: 12 boxes through the 6-slot
                                   # ring, 6 reloaded in the pipelined cast, a ragged last box
                                   # and a partial 64-column tile
                                   (2, 12000, 80)])
@pytest.mark.parametrize("trans", [True, False])
def test_colwise_dense_parity(F, kind, okind, E, R, C, trans):
    x = _bf16((E, R, C), E * 1000 + R + C, 0.02)
    x[0, :, 1] = 0.0
    q, inv = F.fp8moe_quantize_colwise_3d(x.to(DEV), None, trans, kind)
    rq, rinv = OQ.quantize_colwise_3d(_np(x), okind, transpose_out=trans)
    assert np.array_equal(inv.cpu().numpy(), rinv)
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("kind,okind", KINDS)
@pytest.mark.parametrize("sizes", [[96, 0, 0, 928], [30, 0, 47, 23], [4000, 0, 1000], [1, 2, 3, 500, 7],
                                   [0, 0, 64],
                                   # tall and small groups together: the transposed output
                                   # streams slices past the ring (6000: 3000 rows per CTA)
                                   # and fits the rest in it
                                   [6000, 1281, 1280, 33, 0, 2500]])
@pytest.mark.parametrize("trans", [True, False])
def test_colwise_jagged_parity(F, kind, okind, sizes, trans):
    M = sum(sizes)
    C = 48
    x = _bf16((M, C), M + len(sizes), 1.0)
    offs = W.offsets_from_sizes(sizes)
    ot = torch.from_numpy(offs).to(DEV)
    q, inv = F.fp8moe_quantize_colwise_3d(x.to(DEV), ot, trans, kind)
    rq, rinv = OQ.quantize_colwise_jagged(_np(x), offs, okind, transpose_out=trans)
    assert np.array_equal(inv.cpu().numpy(), rinv)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert F.fp8moe_get_device_status() == 0


def test_colwise_jagged_cluster_form():
    """The two-CTA cluster kernel for routed rows (FP8MOE_CW_JAGGED=cluster;
    the one-CTA-per-strip kernel serves them by default) gives identical
    results: the jagged colwise cases rerun with it."""
    import os
    import subprocess
    import sys
    if os.environ.get("FP8MOE_CW_JAGGED"):
        pytest.skip("this process already fixes the jagged kernel")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu",
                        os.path.abspath(__file__), "-k", "colwise_jagged and not cluster_form"],
                       cwd=root, env=dict(os.environ, FP8MOE_CW_JAGGED="cluster"), capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.mark.parametrize("E", [640, 700])
def test_colwise_jagged_many_groups(F, E):
    """Hundreds of routed groups, most of them a fraction of a TMA box, with
    empty and one-row groups among them and one group longer than the ring:
    the transposed kernel's per-group tables, size order and padding."""
    import os
    if os.environ.get("FP8MOE_CW_JAGGED"):
        pytest.skip("this process fixes the jagged colwise kernel")
    rng = np.random.default_rng(E)
    sizes = rng.integers(0, 60, size=E)
    sizes[::7] = 0
    sizes[3::11] = 1
    sizes[5] = 1500
    C = 64
    M = int(sizes.sum())
    x = _bf16((M, C), E, 1.0)
    offs = W.offsets_from_sizes([int(v) for v in sizes])
    q, inv = F.fp8moe_quantize_colwise_3d(x.to(DEV), torch.from_numpy(offs).to(DEV), True, 0)
    assert F.fp8moe_get_device_status() == 0
    rq, rinv = OQ.quantize_colwise_jagged(_np(x), offs, OF.FN, transpose_out=True)
    assert np.array_equal(inv.cpu().numpy(), rinv)
    assert np.array_equal(q.cpu().numpy(), rq)


def test_colwise_jagged_work_counter(F):
    """The routed-rows transposed kernel takes its units from a device work
    counter (one of 16 slots per launch, cleared by the launch's last CTA):
    40 launches in a row (every slot reused), three replays of one captured
    launch (the same slot and tag each time) and two launches in flight at
    once on two streams all give the oracle's codes and scales."""
    import os
    if os.environ.get("FP8MOE_CW_JAGGED"):
        pytest.skip("this process fixes the jagged colwise kernel")
    sizes = [700, 0, 130, 2000, 33, 1, 0, 1600]
    C = 320
    M = sum(sizes)
    x = _bf16((M, C), 91, 1.0)
    offs = W.offsets_from_sizes(sizes)
    rq, rinv = OQ.quantize_colwise_jagged(_np(x), offs, OF.FN, transpose_out=True)
    xd, ot = x.to(DEV), torch.from_numpy(offs).to(DEV)

    def same(q, inv):
        return np.array_equal(q.cpu().numpy(), rq) and np.array_equal(inv.cpu().numpy(), rinv)

    outs = [F.fp8moe_quantize_colwise_3d(xd, ot, True, 0) for _ in range(40)]
    assert F.fp8moe_get_device_status() == 0
    assert all(same(q, inv) for q, inv in outs)
    qs, invs = outs[0][0].clone(), outs[0][1].clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        F.fp8moe_quantize_colwise_3d(xd, ot, True, 0, q=qs, scale_inv=invs)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        F.fp8moe_quantize_colwise_3d(xd, ot, True, 0, q=qs, scale_inv=invs)
    for _ in range(3):
        qs.zero_()
        invs.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert same(qs, invs)
    assert F.fp8moe_get_device_status() == 0
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    q1, i1 = torch.empty_like(qs), torch.empty_like(invs)
    q2, i2 = torch.empty_like(qs), torch.empty_like(invs)
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s1):
        F.fp8moe_quantize_colwise_3d(xd, ot, True, 0, q=q1, scale_inv=i1)
    with torch.cuda.stream(s2):
        F.fp8moe_quantize_colwise_3d(xd, ot, True, 0, q=q2, scale_inv=i2)
    torch.cuda.synchronize()
    assert F.fp8moe_get_device_status() == 0
    assert same(q1, i1) and same(q2, i2)


def test_colwise_jagged_tiny_workload(F):
    wl = W.get_workload("tiny")
    offs = wl.offs()
    x = W.make_activations(wl, "A")
    q, inv = F.fp8moe_quantize_colwise_3d(x.to(DEV), torch.from_numpy(offs).to(DEV), True, 0)
    rq, rinv = OQ.quantize_colwise_jagged(_np(x), offs, OF.FN, transpose_out=True)
    assert np.array_equal(q.cpu().numpy(), rq) and np.array_equal(inv.cpu().numpy(), rinv)


def test_colwise_bad_offsets_set_status(F):
    x = torch.zeros(64, 32, dtype=torch.bfloat16, device=DEV)
    for bad in [[40, 30, 64], [10, 20, 60], [10, 20, 70]]:
        F.fp8moe_quantize_colwise_3d(x, torch.tensor(bad, dtype=torch.int32, device=DEV), True, 0)
        assert F.fp8moe_get_device_status() == 5
    assert F.fp8moe_get_device_status() == 0


# ----------------------------------------------------------------------------
# MXFP8
# ----------------------------------------------------------------------------

def _mx_tie_blocks(rows, C, seed):
    rng = np.random.default_rng(seed)
    tab = OF.decode_table(OF.FN)
    fin = np.sort(tab[np.isfinite(tab) & (tab >= 0)])
    mids = (fin[:-1] + fin[1:]) / 2
    cand = np.concatenate([fin, mids, [464.0, 480.0, 500.0, 0.0]])
    x = rng.choice(cand, size=(rows, C)) * rng.choice([-1.0, 1.0], size=(rows, C))
    blocks = x.reshape(rows, C // 32, 32)
    j = rng.integers(-30, 30, size=(rows, C // 32))
    blocks[..., 0] = 256.0
    x = (blocks * np.ldexp(1.0, j)[..., None]).reshape(rows, C)
    x[0, :32] = 0.0
    x[1, :32] = -0.0
    x[2, 32:64] = np.ldexp(1.0, -133)       # bf16 subnormal block
    t = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(t.float().numpy(), x.astype(np.float32))
    return t


@pytest.mark.parametrize("shape", [(1024, 256), (4, 512, 256), (3, 32), (1, 5120), (333, 96)])
def test_mx_dim0_parity(F, shape):
    x = _bf16(shape, sum(shape), 2.0)
    q, s = F.fp8moe_mxfp8_quantize_dim0(x.to(DEV))
    rq, rs = OQ.mxfp8_quantize_dim0(_np(x))
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


def test_mx_dim0_tie_points(F):
    x = _mx_tie_blocks(64, 256, 3)
    q, s = F.fp8moe_mxfp8_quantize_dim0(x.to(DEV))
    rq, rs = OQ.mxfp8_quantize_dim0(_np(x))
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("shape", [(1024, 256), (4, 512, 256), (32, 16), (96, 80), (160, 128), (1, 256, 5120)])
def test_mx_dim1_parity(F, shape):
    x = _bf16(shape, sum(shape) + 1, 2.0)
    qt, st = F.fp8moe_mxfp8_quantize_dim1(x.to(DEV))
    rqt, rst = OQ.mxfp8_quantize_dim1(_np(x))
    assert np.array_equal(st.cpu().numpy(), rst)
    assert np.array_equal(qt.cpu().numpy(), rqt)


def test_mx_dim1_tie_points(F):
    x = _mx_tie_blocks(256, 64, 4).T.contiguous()    # blocks of 32 along dim 0 after transpose
    qt, st = F.fp8moe_mxfp8_quantize_dim1(x.to(DEV))
    rqt, rst = OQ.mxfp8_quantize_dim1(_np(x))
    assert np.array_equal(st.cpu().numpy(), rst)
    assert np.array_equal(qt.cpu().numpy(), rqt)


def test_mx_tiny_workload(F):
    wl = W.get_workload("tiny")
    for x in [W.make_activations(wl, "A"), W.make_activations(wl, "dY"), W.make_weights(wl, "W1")]:
        q, s = F.fp8moe_mxfp8_quantize_dim0(x.to(DEV))
        rq, rs = OQ.mxfp8_quantize_dim0(_np(x))
        assert np.array_equal(q.cpu().numpy(), rq) and np.array_equal(s.cpu().numpy(), rs)
        qt, st = F.fp8moe_mxfp8_quantize_dim1(x.to(DEV))
        rqt, rst = OQ.mxfp8_quantize_dim1(_np(x))
        assert np.array_equal(qt.cpu().numpy(), rqt) and np.array_equal(st.cpu().numpy(), rst)


# ----------------------------------------------------------------------------
# swizzle
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("B,R,Cs", [(1, 1024, 8), (4, 512, 8), (1, 1, 1), (2, 200, 7), (1, 300, 160),
                                    # rows of whole 16-byte chunks (the 16-byte staging path):
                                    # batched with a ragged row block, two full column chunks
                                    (3, 257, 48), (1, 128, 256)])
def test_swizzle_plain(F, B, R, Cs):
    s = torch.randint(1, 255, (B, R, Cs), dtype=torch.uint8, generator=torch.Generator().manual_seed(R))
    out = F.fp8moe_swizzle_scales_128x4(s.to(DEV))
    ref = OS.swizzle(s.numpy() if B > 1 else s[0].numpy())
    assert np.array_equal(out.cpu().numpy(), ref)


@pytest.mark.parametrize("sizes", [[96, 0, 0, 928], [100, 0, 160, 40], [0, 0, 5], [300]])
@pytest.mark.parametrize("Cs", [6, 32])
def test_swizzle_group_rows(F, sizes, Cs):
    R = sum(sizes)
    s = torch.randint(1, 255, (R, Cs), dtype=torch.uint8, generator=torch.Generator().manual_seed(R))
    offs = W.offsets_from_sizes(sizes)
    out = F.fp8moe_swizzle_scales_128x4(s.to(DEV), torch.from_numpy(offs).to(DEV), F.GROUP_ROWS)
    assert np.array_equal(out.cpu().numpy(), OS.swizzle(s.numpy(), offs, OS.GROUP_ROWS))


@pytest.mark.parametrize("sizes", [[96, 0, 0, 928], [64, 0, 256], [32], [0, 320]])
def test_swizzle_group_cols(F, sizes):
    M = sum(sizes)
    s = torch.randint(1, 255, (130, M // 32), dtype=torch.uint8, generator=torch.Generator().manual_seed(M))
    offs = W.offsets_from_sizes(sizes)
    out = F.fp8moe_swizzle_scales_128x4(s.to(DEV), torch.from_numpy(offs).to(DEV), F.GROUP_COLS)
    assert np.array_equal(out.cpu().numpy(), OS.swizzle(s.numpy(), offs, OS.GROUP_COLS))


def test_swizzle_bad_offsets_set_status(F):
    s = torch.ones(64, 4, dtype=torch.uint8, device=DEV)
    F.fp8moe_swizzle_scales_128x4(s, torch.tensor([40, 30, 64], dtype=torch.int32, device=DEV), F.GROUP_ROWS)
    assert F.fp8moe_get_device_status() == 5
    F.fp8moe_swizzle_scales_128x4(s, torch.tensor([40, 64], dtype=torch.int32, device=DEV), F.GROUP_COLS)
    assert F.fp8moe_get_device_status() == 5     # 40 is not a multiple of 32
    # rows of whole 16-byte chunks: the bulk-copy kernel
    s32 = torch.ones(64, 32, dtype=torch.uint8, device=DEV)
    F.fp8moe_swizzle_scales_128x4(s32, torch.tensor([40, 30, 64], dtype=torch.int32, device=DEV), F.GROUP_ROWS)
    assert F.fp8moe_get_device_status() == 5
    assert F.fp8moe_get_device_status() == 0


# ----------------------------------------------------------------------------
# dual-direction MXFP8 with scales written in their final layout
# ----------------------------------------------------------------------------

def _mx_ref(x_np):
    q0, s0 = OQ.mxfp8_quantize_dim0(x_np)
    q1, s1 = OQ.mxfp8_quantize_dim1(x_np)
    return q0, s0, q1, s1


@pytest.mark.parametrize("shape", [(1024, 256), (96, 96), (32, 64), (160, 5120),
                                   # a last 128-column tile with one 64-column box in range
                                   (32, 192), (64, 448)])
def test_mx_dual_rowmajor(F, shape):
    x = _bf16(shape, sum(shape) + 7, 2.0)
    q0, s0, q1, s1 = F.fp8moe_mxfp8_quantize_dual(x.to(DEV), None, F.SCALES_ROWMAJOR, F.SCALES_ROWMAJOR)
    r0, rs0, r1, rs1 = _mx_ref(_np(x))
    assert np.array_equal(q0.cpu().numpy(), r0) and np.array_equal(s0.cpu().numpy(), rs0)
    assert np.array_equal(q1.cpu().numpy(), r1) and np.array_equal(s1.cpu().numpy(), rs1)


@pytest.mark.parametrize("shape", [(4, 512, 256), (3, 96, 160), (1, 256, 5120)])
def test_mx_dual_batched_swizzled(F, shape):
    x = _bf16(shape, sum(shape) + 8, 0.05)
    q0, s0, q1, s1 = F.fp8moe_mxfp8_quantize_dual(x.to(DEV), None, F.NO_GROUPS, F.NO_GROUPS)
    r0, rs0, r1, rs1 = _mx_ref(_np(x))
    assert np.array_equal(q0.cpu().numpy(), r0)
    assert np.array_equal(q1.cpu().numpy(), r1)
    assert np.array_equal(s0.cpu().numpy(), OS.swizzle(rs0))
    assert np.array_equal(s1.cpu().numpy(), OS.swizzle(rs1))


@pytest.mark.parametrize("sizes", [[96, 0, 0, 928], [64, 0, 352, 32, 160], [0, 0, 64], [32]])
def test_mx_dual_grouped(F, sizes):
    M = int(sum(sizes))
    x = _bf16((M, 192), M + 9, 1.5)
    offs = W.offsets_from_sizes(sizes)
    q0, s0, q1, s1 = F.fp8moe_mxfp8_quantize_dual(x.to(DEV), torch.from_numpy(offs).to(DEV), F.GROUP_ROWS,
                                                  F.GROUP_COLS)
    r0, rs0, r1, rs1 = _mx_ref(_np(x))
    assert np.array_equal(q0.cpu().numpy(), r0)
    assert np.array_equal(q1.cpu().numpy(), r1)
    assert np.array_equal(s0.cpu().numpy(), OS.swizzle(rs0, offs, OS.GROUP_ROWS))
    assert np.array_equal(s1.cpu().numpy(), OS.swizzle(rs1, offs, OS.GROUP_COLS))
    assert F.fp8moe_get_device_status() == 0


def test_mx_dual_single_direction(F):
    x = _bf16((256, 128), 5, 1.0)
    q0, s0, q1, s1 = F.fp8moe_mxfp8_quantize_dual(x.to(DEV), None, F.SCALES_ROWMAJOR, F.NO_GROUPS, dim1=False)
    r0, rs0, _, _ = _mx_ref(_np(x))
    assert q1 is None and np.array_equal(q0.cpu().numpy(), r0) and np.array_equal(s0.cpu().numpy(), rs0)
    q0, s0, q1, s1 = F.fp8moe_mxfp8_quantize_dual(x.to(DEV), None, F.NO_GROUPS, F.SCALES_ROWMAJOR, dim0=False)
    _, _, r1, rs1 = _mx_ref(_np(x))
    assert q0 is None and np.array_equal(q1.cpu().numpy(), r1) and np.array_equal(s1.cpu().numpy(), rs1)


def test_mx_dual_tie_points(F):
    x = _mx_tie_blocks(256, 256, 6)
    q0, s0, q1, s1 = F.fp8moe_mxfp8_quantize_dual(x.to(DEV), None, F.SCALES_ROWMAJOR, F.SCALES_ROWMAJOR)
    r0, rs0, r1, rs1 = _mx_ref(_np(x))
    assert np.array_equal(q0.cpu().numpy(), r0) and np.array_equal(s0.cpu().numpy(), rs0)
    assert np.array_equal(q1.cpu().numpy(), r1) and np.array_equal(s1.cpu().numpy(), rs1)


def test_mx_dual_bad_offsets(F):
    x = torch.zeros(128, 64, dtype=torch.bfloat16, device=DEV)
    F.fp8moe_mxfp8_quantize_dual(x, torch.tensor([64, 32, 128], dtype=torch.int32, device=DEV), F.GROUP_ROWS,
                                 F.GROUP_COLS)
    assert F.fp8moe_get_device_status() == 5
    assert F.fp8moe_get_device_status() == 0


@pytest.mark.parametrize("l0,l1", [("SCALES_ROWMAJOR", "GROUP_COLS"), ("GROUP_ROWS", "SCALES_ROWMAJOR"),
                                   ("GROUP_ROWS", "NO_GROUPS"), ("NO_GROUPS", "GROUP_COLS")])
def test_mx_dual_mixed_layouts(F, l0, l1):
    """Each direction's scales in its own layout; all-zero blocks (scale byte
    0, codes 0) in both directions."""
    sizes = [64, 0, 160, 32]
    offs = W.offsets_from_sizes(sizes)
    x = _bf16((256, 320), 31, 1.0)
    x[32:64, :] = 0.0          # zero dim1 blocks (and dim0 rows)
    x[:, 96:128] = 0.0         # zero dim0 blocks
    q0, s0, q1, s1 = F.fp8moe_mxfp8_quantize_dual(x.to(DEV), torch.from_numpy(offs).to(DEV), getattr(F, l0),
                                                  getattr(F, l1))
    r0, rs0, r1, rs1 = _mx_ref(_np(x))

    def lay(rs, name, axis):
        if name == "SCALES_ROWMAJOR":
            return rs
        if name == "NO_GROUPS":
            return OS.swizzle(rs)
        return OS.swizzle(rs, offs, axis)

    assert np.array_equal(q0.cpu().numpy(), r0) and np.array_equal(q1.cpu().numpy(), r1)
    assert np.array_equal(s0.cpu().numpy(), lay(rs0, l0, OS.GROUP_ROWS))
    assert np.array_equal(s1.cpu().numpy(), lay(rs1, l1, OS.GROUP_COLS))
    assert F.fp8moe_get_device_status() == 0


@pytest.mark.parametrize("C", [96, 256])
def test_mx_dual_unaligned_row_groups(F, C):
    """dim0 scales grouped by rows whose groups start off 16-row boundaries
    (allowed when dim1's scales are not grouped); 256 columns take the
    warp-specialised kernel, where a 32-row sub-tile that holds two groups
    gives each row its own group."""
    sizes = [40, 0, 200, 8, 72]          # sums to 320
    offs = W.offsets_from_sizes(sizes)
    x = _bf16((320, C), 41, 1.0)
    q0, s0, q1, s1 = F.fp8moe_mxfp8_quantize_dual(x.to(DEV), torch.from_numpy(offs).to(DEV), F.GROUP_ROWS,
                                                  F.SCALES_ROWMAJOR)
    r0, rs0, r1, rs1 = _mx_ref(_np(x))
    assert np.array_equal(q0.cpu().numpy(), r0) and np.array_equal(q1.cpu().numpy(), r1)
    assert np.array_equal(s0.cpu().numpy(), OS.swizzle(rs0, offs, OS.GROUP_ROWS))
    assert np.array_equal(s1.cpu().numpy(), rs1)
    assert F.fp8moe_get_device_status() == 0


def test_mx_dual_unaligned_scale_buffers(F):
    """Scale buffers at odd byte offsets (views into larger buffers) and
    row-major scales whose rows are not a multiple of 4 bytes."""
    x = _bf16((160, 96), 51, 1.0)                 # C/32 = 3, R/32 = 5
    r0, rs0, r1, rs1 = _mx_ref(_np(x))
    big0 = torch.zeros(160 * 3 + 8, dtype=torch.uint8, device=DEV)
    big1 = torch.zeros(96 * 5 + 8, dtype=torch.uint8, device=DEV)
    s0 = big0[1:1 + 160 * 3].view(160, 3)
    s1 = big1[3:3 + 96 * 5].view(96, 5)
    q0, _, q1, _ = F.fp8moe_mxfp8_quantize_dual(x.to(DEV), None, F.SCALES_ROWMAJOR, F.SCALES_ROWMAJOR, s0=s0,
                                                s1=s1)
    assert np.array_equal(q0.cpu().numpy(), r0) and np.array_equal(q1.cpu().numpy(), r1)
    assert np.array_equal(s0.cpu().numpy(), rs0) and np.array_equal(s1.cpu().numpy(), rs1)
    qt, st = F.fp8moe_mxfp8_quantize_dim1(x.to(DEV))
    assert np.array_equal(qt.cpu().numpy(), r1) and np.array_equal(st.cpu().numpy(), rs1)
    assert F.fp8moe_get_device_status() == 0


@pytest.mark.parametrize("band", ["4", "2"])
def test_mx_dual_band_heights(band):
    """The fused kernel's band heights (chosen by tensor size) give identical
    results: the dual / dim1 cases rerun with the height fixed."""
    import os
    import subprocess
    import sys
    if os.environ.get("FP8MOE_DUAL_BAND") or os.environ.get("FP8MOE_DUAL_PREFETCH"):
        pytest.skip("this process already fixes the band height or the load form")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu",
                        os.path.abspath(__file__), "-k",
                        "(mx_dual or mx_dim1) and not band_heights and not warp_specialised"],
                       cwd=root, env=dict(os.environ, FP8MOE_DUAL_BAND=band), capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


def test_mx_dim1_warp_specialised_form():
    """The warp-specialised kernel's dim1-only instance (selected with
    FP8MOE_DUAL_WS=1; the register-tile form serves that case by default)
    gives identical results: the dim1 and dual cases rerun with it."""
    import os
    import subprocess
    import sys
    if os.environ.get("FP8MOE_DUAL_WS") or os.environ.get("FP8MOE_DUAL_PREFETCH") or os.environ.get("FP8MOE_DUAL_BAND"):
        pytest.skip("this process already fixes the kernel form")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu",
                        os.path.abspath(__file__), "-k",
                        "(mx_dual or mx_dim1) and not band_heights and not load_forms and not warp_specialised"],
                       cwd=root, env=dict(os.environ, FP8MOE_DUAL_WS="1"), capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.mark.parametrize("prefetch", ["0", "1"])
def test_mx_dual_load_forms(prefetch):
    """The register-tile form of the fused kernel (the one for fewer than 128
    columns; FP8MOE_DUAL_WS=0 selects it for every shape) in both ways it gets
    its sub-tiles (a TMA load into the warp's buffer one sub-tile ahead, or
    plain loads into registers; chosen by tensor size) gives identical
    results: the dual / dim1 cases rerun with that form and the load fixed."""
    import os
    import subprocess
    import sys
    if os.environ.get("FP8MOE_DUAL_PREFETCH") or os.environ.get("FP8MOE_DUAL_BAND"):
        pytest.skip("this process already fixes the load form or the band height")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu",
                        os.path.abspath(__file__), "-k",
                        "(mx_dual or mx_dim1) and not band_heights and not load_forms and not warp_specialised"],
                       cwd=root, env=dict(os.environ, FP8MOE_DUAL_PREFETCH=prefetch, FP8MOE_DUAL_WS="0"),
                       capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


# ----------------------------------------------------------------------------
# timeout path of the warp-specialised quantizers (no GPU fault: a load that
# is never issued)
# ----------------------------------------------------------------------------

def test_quant_ring_timeout_dual(F):
    """The one-shot testing hook makes the first CTA of the next
    warp-specialised dual-direction launch never load its first sub-tile:
    that CTA's consumer warps' bounded wait (2 s) runs out, the launch
    reports FP8MOE_ERR_TIMEOUT, its producer still waits for the loads it
    issued, and the next call (the hook is spent) is exact."""
    import os
    if os.environ.get("FP8MOE_DUAL_WS"):
        pytest.skip("this process fixes the dual kernel form")
    x = _bf16((256, 512), 91, 1.0)
    F.fp8moe_testing_stall_next_quant_ring()
    F.fp8moe_mxfp8_quantize_dual(x.to(DEV), None, F.SCALES_ROWMAJOR, F.SCALES_ROWMAJOR)
    assert F.fp8moe_get_device_status() == 6          # FP8MOE_ERR_TIMEOUT
    q0, s0, q1, s1 = F.fp8moe_mxfp8_quantize_dual(x.to(DEV), None, F.SCALES_ROWMAJOR, F.SCALES_ROWMAJOR)
    assert F.fp8moe_get_device_status() == 0
    r0, rs0, r1, rs1 = _mx_ref(_np(x))
    assert np.array_equal(q0.cpu().numpy(), r0) and np.array_equal(s0.cpu().numpy(), rs0)
    assert np.array_equal(q1.cpu().numpy(), r1) and np.array_equal(s1.cpu().numpy(), rs1)


def test_quant_ring_timeout_jagged(F):
    """The same hook on the routed-rows transposed colwise kernel: the first
    box of unit 0 (the largest group's first strip, whichever CTA takes it)
    is counted as issued but never loaded, so the consumer group waiting for
    it runs out (2 s) while the other group and the other CTAs carry on;
    FP8MOE_ERR_TIMEOUT, then an exact call."""
    import os
    if os.environ.get("FP8MOE_CW_JAGGED"):
        pytest.skip("this process fixes the jagged colwise kernel")
    sizes = [96, 0, 320, 32, 160]
    offs = W.offsets_from_sizes(sizes)
    x = _bf16((int(sum(sizes)), 192), 17, 0.5)
    ot = torch.from_numpy(offs).to(DEV)
    F.fp8moe_testing_stall_next_quant_ring()
    F.fp8moe_quantize_colwise_3d(x.to(DEV), ot, True, 0)
    assert F.fp8moe_get_device_status() == 6          # FP8MOE_ERR_TIMEOUT
    q, inv = F.fp8moe_quantize_colwise_3d(x.to(DEV), ot, True, 0)
    assert F.fp8moe_get_device_status() == 0
    rq, rinv = OQ.quantize_colwise_jagged(_np(x), offs, OF.FN, transpose_out=True)
    assert np.array_equal(inv.cpu().numpy(), rinv)
    assert np.array_equal(q.cpu().numpy(), rq)
