"""Full-size parity on the real workload shapes, on sampled outputs.

The GPU runs the whole path at the configuration sizes, in the launch
configuration bench.py times (fused dual-direction MXFP8 quantization with
scales written in their final layout, then the grouped GEMMs).  The oracle
recomputes sampled outputs one by one from the bf16 inputs: quantized codes
and scales of sampled rows / column slices must match bit for bit; sampled
GEMM outputs must satisfy |gpu - ref| <= 8e-3 |ref| + 1e-3 sum_k |a_k b_k|.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats as OF, quant as OQ, swizzle as OS

pytestmark = pytest.mark.gpu
DEV = "cuda"
RTOL, BTOL = 8e-3, 1e-3


@pytest.fixture(scope="module")
def F():
    from mxfp8_moe_quantization_gb300 import build as B
    B.build()
    import mxfp8_moe_quantization_gb300 as m
    return m


def _np(t):
    return t.float().cpu().numpy()


def _check_vals(got, ref, bound, what):
    err = np.abs(got - ref)
    lim = RTOL * np.abs(ref) + BTOL * bound
    assert np.all(err <= lim), f"{what}: worst excess {float((err - lim).max())}"


def _mx_rows(x_rows):
    """Oracle MXFP8 dequantized rows (dim0 blocks along the row)."""
    q, s = OQ.mxfp8_quantize_dim0(x_rows)
    return OQ.dequant_mx(q, s)


def _mx_cols(x_cols):
    """Oracle MXFP8 dequantized columns of x [R, c] (dim1 blocks along R)."""
    qt, st = OQ.mxfp8_quantize_dim1(x_cols)
    return OQ.dequant_mx(qt, st)          # [c, R]


def _sample_rows(offs, rng, per_group=2):
    starts, ends = OQ.group_bounds(offs)
    rows = []
    for e in range(len(offs)):
        if ends[e] > starts[e]:
            rows += [int(starts[e]), int(ends[e] - 1)]
            rows += list(rng.integers(starts[e], ends[e], size=per_group))
    return np.array(sorted(set(rows)))


# the operands of each expert weight: (activation, gradient, weight); W1
# [E, N, K] takes A [M, K] and dY [M, N]; W2 [E, K, N] takes A2 [M, N] and
# dY2 [M, K]
OPERANDS = {"W1": ("A", "dY", "W1"), "W2": ("A2", "dY2", "W2")}


def _layer(wl, which, dev):
    an, dn, wn = OPERANDS[which]
    a = W.make_activations(wl, an, device=dev)
    dy = W.make_activations(wl, dn, device=dev)
    w = W.make_weights(wl, wn, device=dev)
    return a, dy, w


def _swz_rows_bytes(buf, offs_np, rows, ncols, E):
    """Bytes of a row-grouped swizzled scale buffer (GROUP_ROWS) at the
    given rows, all ``ncols`` scale columns: [len(rows), ncols]."""
    R = int(offs_np[-1])
    _, Cp = OS.swizzled_shape(R, ncols, E, OS.GROUP_ROWS)
    starts, ends = OQ.group_bounds(offs_np)
    P = OQ.padded_starts(offs_np, 128)
    g = np.searchsorted(ends, rows, side="right")
    prow = P[g] + (rows - starts[g])
    o = OS.tile_offset(prow[:, None], np.arange(ncols)[None, :], Cp)
    return buf.cpu().numpy()[o]


def _swz_cols_bytes(buf, offs_np, rows, nscols, E):
    """Bytes of a column-grouped swizzled scale buffer (GROUP_COLS, offsets
    over the contracting elements) at the given rows, every real scale
    column: [len(rows), nscols]."""
    _, Cp = OS.swizzled_shape(len(rows), nscols, E, OS.GROUP_COLS)
    sc = np.asarray(offs_np, dtype=np.int64) // 32
    starts, ends = OQ.group_bounds(sc)
    Q = OQ.padded_starts(sc, 4)
    cols = np.arange(nscols)
    g = np.searchsorted(ends, cols, side="right")
    pcol = Q[g] + (cols - starts[g])
    o = OS.tile_offset(np.asarray(rows)[:, None], pcol[None, :], Cp)
    return buf.cpu().numpy()[o]


def _swz_batch_bytes(buf, R, ncols, b, rows):
    """Bytes of batch ``b`` of a plain per-batch swizzled buffer (NO_GROUPS)
    at the given rows: [len(rows), ncols]."""
    Rp, Cp = OS.swizzled_shape(R, ncols)
    o = b * Rp * Cp + OS.tile_offset(np.asarray(rows)[:, None], np.arange(ncols)[None, :], Cp)
    return buf.cpu().numpy()[o]


@pytest.mark.parametrize("which", ["W1", "W2"])
@pytest.mark.parametrize("name", ["scout", "dsv3"])
def test_mxfp8_fullsize(F, name, which):
    wl = W.get_workload(name)
    rng = np.random.default_rng(7)
    a, dy, w = _layer(wl, which, DEV)
    M = wl.M
    E, N, K = w.shape                       # this weight's GEMM: [M, K] x [E, N, K]^T
    offs_np = wl.offs()
    offs = torch.from_numpy(offs_np).to(DEV)
    qa, sa, qat, sat = F.fp8moe_mxfp8_quantize_dual(a, offs, F.GROUP_ROWS, F.GROUP_COLS)
    qw, sw, qwt, swt = F.fp8moe_mxfp8_quantize_dual(w, None, F.NO_GROUPS, F.NO_GROUPS)
    qdy, sdy, qdyt, sdyt = F.fp8moe_mxfp8_quantize_dual(dy, offs, F.GROUP_ROWS, F.GROUP_COLS)
    out = F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, qa, sa, qw, sw, offs)
    da = F.fp8moe_scaled_grouped_mm_dgrad(F.MXFP8, qdy, sdy, qwt, swt, offs)
    dw = F.fp8moe_scaled_grouped_mm_wgrad(F.MXFP8, qdyt, sdyt, qat, sat, offs, M)
    torch.cuda.synchronize()
    assert F.fp8moe_get_device_status() == 0

    rows = _sample_rows(offs_np, rng)
    rt = torch.from_numpy(rows).to(DEV)
    starts, ends = OQ.group_bounds(offs_np)
    grp = np.searchsorted(ends, rows, side="right")
    # codes and e8m0 scale bytes of sampled rows (dim0, row-grouped 128x4
    # layout) and of a column slice (dim1, column-grouped layout), for the
    # activation and the gradient
    for x, q0, s0, q1, s1, C in [(a, qa, sa, qat, sat, K), (dy, qdy, sdy, qdyt, sdyt, N)]:
        rq, rs = OQ.mxfp8_quantize_dim0(_np(x[rt]))
        assert np.array_equal(q0[rt].cpu().numpy(), rq)
        assert np.array_equal(_swz_rows_bytes(s0, offs_np, rows, C // 32, E), rs)
        c0 = int(rng.integers(0, C // 64)) * 64
        rqt, rst = OQ.mxfp8_quantize_dim1(_np(x[:, c0:c0 + 64]))
        assert np.array_equal(q1[c0:c0 + 64].cpu().numpy(), rqt)
        got = _swz_cols_bytes(s1, offs_np, np.arange(c0, c0 + 64), M // 32, E)
        assert np.array_equal(got, rst)
    # weight codes and scales: sampled rows (dim0) and a column slice (dim1)
    # of a few experts, the last one included
    for e in sorted(set(rng.integers(0, E, size=2).tolist() + [E - 1])):
        wr = np.array(sorted(set(rng.integers(0, N, size=8).tolist() + [0, N - 1])))
        rq, rs = OQ.mxfp8_quantize_dim0(_np(w[e][torch.from_numpy(wr).to(DEV)]))
        assert np.array_equal(qw[e][torch.from_numpy(wr).to(DEV)].cpu().numpy(), rq)
        assert np.array_equal(_swz_batch_bytes(sw, N, K // 32, e, wr), rs)
        k0 = int(rng.integers(0, K // 64)) * 64
        rqt, rst = OQ.mxfp8_quantize_dim1(_np(w[e][:, k0:k0 + 64]))
        assert np.array_equal(qwt[e][k0:k0 + 64].cpu().numpy(), rqt)
        assert np.array_equal(_swz_batch_bytes(swt, K, N // 32, e, np.arange(k0, k0 + 64)), rst)

    # forward: sampled rows x sampled columns
    a_rows = _np(a[rt])
    ncols = np.array(sorted(set(rng.integers(0, N, size=24).tolist() + [0, N - 1])))
    a_deq = _mx_rows(a_rows)
    got = _np(out[rt][:, torch.from_numpy(ncols).to(DEV)])
    ref = np.zeros_like(got, dtype=np.float64)
    bnd = np.zeros_like(ref)
    for e in np.unique(grp):
        sel = grp == e
        w_deq = _mx_rows(_np(w[int(e)][torch.from_numpy(ncols).to(DEV)]))
        ref[sel] = a_deq[sel] @ w_deq.T
        bnd[sel] = np.abs(a_deq[sel]) @ np.abs(w_deq).T
    _check_vals(got, ref, bnd, f"{name} {which} fwd")

    # dgrad: sampled rows x sampled K columns (W quantized along N)
    kcols = np.array(sorted(set(rng.integers(0, K, size=16).tolist() + [K - 1])))
    dy_deq = _mx_rows(_np(dy[rt]))
    got = _np(da[rt][:, torch.from_numpy(kcols).to(DEV)])
    ref = np.zeros_like(got, dtype=np.float64)
    bnd = np.zeros_like(ref)
    for e in np.unique(grp):
        sel = grp == e
        wt_deq = _mx_cols(_np(w[int(e)][:, torch.from_numpy(kcols).to(DEV)]))   # [k, N]
        ref[sel] = dy_deq[sel] @ wt_deq.T
        bnd[sel] = np.abs(dy_deq[sel]) @ np.abs(wt_deq).T
    _check_vals(got, ref, bnd, f"{name} {which} dgrad")

    # wgrad: a few (n, k) of every expert, empty experts exactly zero
    nn = rng.integers(0, N, size=6)
    kk = rng.integers(0, K, size=6)
    nt, kt = torch.from_numpy(nn).to(DEV), torch.from_numpy(kk).to(DEV)
    for e in range(E):
        s0, s1 = int(starts[e]), int(ends[e])
        got = _np(dw[e][nt][:, kt])
        if s1 == s0:
            assert np.all(got == 0)
            continue
        dyc = _mx_cols(_np(dy[s0:s1][:, nt]))      # [6, g]
        ac = _mx_cols(_np(a[s0:s1][:, kt]))        # [6, g]
        _check_vals(got, dyc @ ac.T, np.abs(dyc) @ np.abs(ac).T, f"{name} {which} wgrad e={e}")


def test_dsv3_expert_weight_quantization_fullsize(F):
    """The DeepSeek-V3 layer's standalone MXFP8 quantization of all expert
    weights (W1 [256, 2048, 7168] and W2 [256, 7168, 2048], both directions,
    scales in the 128x4 layout per expert), as bench.py times it: every code
    and scale byte of a seeded sample of whole experts of both weights is
    compared bit for bit with the oracle."""
    wl = W.get_workload("dsv3")
    rng = np.random.default_rng(29)
    for which in ["W1", "W2"]:
        w = W.make_weights(wl, which, device=DEV)
        E, R, C = w.shape
        q0, s0, q1, s1 = F.fp8moe_mxfp8_quantize_dual(w, None, F.NO_GROUPS, F.NO_GROUPS)
        torch.cuda.synchronize()
        assert F.fp8moe_get_device_status() == 0
        Rp0, Cp0 = OS.swizzled_shape(R, C // 32)
        Rp1, Cp1 = OS.swizzled_shape(C, R // 32)
        for e in sorted(set(rng.integers(0, E - 1, size=1).tolist() + [E - 1])):
            x = _np(w[e])
            rq, rs = OQ.mxfp8_quantize_dim0(x)
            assert np.array_equal(q0[e].cpu().numpy(), rq), (which, e, "dim0 codes")
            assert np.array_equal(s0[e * Rp0 * Cp0:(e + 1) * Rp0 * Cp0].cpu().numpy(), OS.swizzle(rs)), \
                (which, e, "dim0 scales")
            rqt, rst = OQ.mxfp8_quantize_dim1(x)
            assert np.array_equal(q1[e].cpu().numpy(), rqt), (which, e, "dim1 codes")
            assert np.array_equal(s1[e * Rp1 * Cp1:(e + 1) * Rp1 * Cp1].cpu().numpy(), OS.swizzle(rst)), \
                (which, e, "dim1 scales")
        del w, q0, s0, q1, s1
        torch.cuda.empty_cache()


@pytest.mark.parametrize("name,which", [("llama3_8b", "W1"), ("dsmoe_16b", "W1"), ("dsmoe_16b", "W2")])
def test_rowwise_fullsize(F, name, which):
    wl = W.get_workload(name)
    rng = np.random.default_rng(11)
    a, dy, w = _layer(wl, which, DEV)
    M = wl.M
    E, N, K = w.shape
    offs_np = wl.offs()
    offs = torch.from_numpy(offs_np).to(DEV)
    qa, ia = F.fp8moe_quantize_rowwise(a)
    qw, iw = F.fp8moe_quantize_rowwise(w.reshape(E * N, K))
    qdy, idy = F.fp8moe_quantize_rowwise(dy)
    qwt, iwt = F.fp8moe_quantize_colwise_3d(w, None, True)          # [E, K, N]
    qdyt, idyt = F.fp8moe_quantize_colwise_3d(dy, offs, True)       # [N, Mt]
    qat, iat = F.fp8moe_quantize_colwise_3d(a, offs, True)          # [K, Mt]
    out = F.fp8moe_scaled_grouped_mm_fwd(F.ROWWISE, qa, ia, qw.view(E, N, K), iw.view(E, N), offs)
    da = F.fp8moe_scaled_grouped_mm_dgrad(F.ROWWISE, qdy, idy, qwt, iwt, offs)
    dw = F.fp8moe_scaled_grouped_mm_wgrad(F.ROWWISE, qdyt, idyt, qat, iat, offs, M)
    torch.cuda.synchronize()
    assert F.fp8moe_get_device_status() == 0

    rows = _sample_rows(offs_np, rng, 1)
    starts, ends = OQ.group_bounds(offs_np)
    grp = np.searchsorted(ends, rows, side="right")
    rt = torch.from_numpy(rows).to(DEV)
    qr, ir = OQ.quantize_rowwise(_np(a[rt]))
    assert np.array_equal(qa[rt].cpu().numpy(), qr) and np.array_equal(ia[rt].cpu().numpy(), ir)
    a_deq = OQ.dequant_rows(qr, ir)
    ncols = np.array(sorted(set(rng.integers(0, N, size=16).tolist())))
    nt = torch.from_numpy(ncols).to(DEV)
    got = _np(out[rt][:, nt])
    ref = np.zeros_like(got, dtype=np.float64)
    bnd = np.zeros_like(ref)
    for e in np.unique(grp):
        sel = grp == e
        wq, wi = OQ.quantize_rowwise(_np(w[int(e)][nt]))
        wd = OQ.dequant_rows(wq, wi)
        ref[sel] = a_deq[sel] @ wd.T
        bnd[sel] = np.abs(a_deq[sel]) @ np.abs(wd).T
    _check_vals(got, ref, bnd, f"{name} {which} fwd")

    kcols = np.array(sorted(set(rng.integers(0, K, size=8).tolist())))
    kt = torch.from_numpy(kcols).to(DEV)
    dq, di = OQ.quantize_rowwise(_np(dy[rt]))
    dy_deq = OQ.dequant_rows(dq, di)
    got = _np(da[rt][:, kt])
    ref = np.zeros_like(got, dtype=np.float64)
    bnd = np.zeros_like(ref)
    for e in np.unique(grp):
        sel = grp == e
        cq, ci = OQ.quantize_colwise_3d(_np(w[int(e)][:, kt])[None], transpose_out=True)   # [1, k, N]
        wt = OF.decode(cq[0]) * ci[0][:, None].astype(np.float64)
        assert np.array_equal(qwt[int(e)][kt].cpu().numpy(), cq[0])
        ref[sel] = dy_deq[sel] @ wt.T
        bnd[sel] = np.abs(dy_deq[sel]) @ np.abs(wt).T
    _check_vals(got, ref, bnd, f"{name} {which} dgrad")

    # the jagged transposed codes of the activation (the wgrad operand), bit
    # for bit on sampled columns of every group: each group at its padded
    # start, its padding and the slack after the last group zero
    P = OQ.padded_starts(offs_np, 32)
    kc = np.array(sorted(set([0, K - 1] + rng.integers(0, K, size=4).tolist())))
    qat_np = qat[torch.from_numpy(kc).to(DEV)].cpu().numpy()
    iat_np = iat.cpu().numpy()
    for e in range(E):
        s0, s1 = int(starts[e]), int(ends[e])
        if s1 == s0:
            continue
        rq_, ri_ = OQ.quantize_colwise_3d(_np(a[s0:s1][:, torch.from_numpy(kc).to(DEV)])[None], transpose_out=True)
        assert np.array_equal(qat_np[:, P[e]:P[e] + (s1 - s0)], rq_[0]), f"{name} jagged codes e={e}"
        assert not qat_np[:, P[e] + (s1 - s0):P[e] + (s1 - s0 + 31) // 32 * 32].any(), f"padding e={e}"
        assert np.array_equal(iat_np[e][kc], ri_[0]), f"{name} jagged scales e={e}"
    last = int(ends[-1] - starts[-1])
    assert not qat_np[:, P[-1] + (last + 31) // 32 * 32:].any(), "slack after the last group"

    nn = torch.from_numpy(rng.integers(0, N, size=4)).to(DEV)
    kk = torch.from_numpy(rng.integers(0, K, size=4)).to(DEV)
    for e in range(E):
        s0, s1 = int(starts[e]), int(ends[e])
        got = _np(dw[e][nn][:, kk])
        if s1 == s0:
            assert np.all(got == 0)
            continue
        dq, di = OQ.quantize_colwise_3d(_np(dy[s0:s1][:, nn])[None], transpose_out=True)
        aq, ai = OQ.quantize_colwise_3d(_np(a[s0:s1][:, kk])[None], transpose_out=True)
        dyc = OF.decode(dq[0]) * di[0][:, None].astype(np.float64)
        ac = OF.decode(aq[0]) * ai[0][:, None].astype(np.float64)
        _check_vals(got, dyc @ ac.T, np.abs(dyc) @ np.abs(ac).T, f"{name} {which} wgrad e={e}")


def test_blockwise_fullsize(F):
    """Blockwise recipe on the Llama4-Scout layer (W1 [16, 8192, 5120], 16,640
    routed rows): the GPU quantizes every operand and runs the three GEMMs;
    the oracle recomputes sampled row tiles, weight tiles, token tiles and
    sampled outputs from the bf16 inputs alone."""
    from oracle import blockwise as OB
    wl = W.get_workload("scout")
    rng = np.random.default_rng(13)
    M, E, N, K = wl.M, wl.E, wl.N, wl.K
    offs_np = wl.offs()
    offs = torch.from_numpy(offs_np).to(DEV)
    a = W.make_activations(wl, "A", device=DEV)
    dy = W.make_activations(wl, "dY", device=DEV)
    w = W.make_weights(wl, "W1", device=DEV)
    qa, sa = F.fp8moe_quantize_blockwise_rows(a)
    qw, qwt, sw = F.fp8moe_quantize_blockwise_weight(w)
    qdy, sdy = F.fp8moe_quantize_blockwise_rows(dy)
    qdyt, sdyt = F.fp8moe_quantize_blockwise_tokens(dy, offs)
    qat, sat = F.fp8moe_quantize_blockwise_tokens(a, offs)
    out = F.fp8moe_scaled_grouped_mm_fwd(F.BLOCKWISE, qa, sa, qw, sw, offs)
    da = F.fp8moe_scaled_grouped_mm_dgrad(F.BLOCKWISE, qdy, sdy, qwt, sw, offs)
    dw = F.fp8moe_scaled_grouped_mm_wgrad(F.BLOCKWISE, qdyt, sdyt, qat, sat, offs, M)
    torch.cuda.synchronize()
    assert F.fp8moe_get_device_status() == 0

    rows = _sample_rows(offs_np, rng, 1)
    starts, ends = OQ.group_bounds(offs_np)
    grp = np.searchsorted(ends, rows, side="right")
    rt = torch.from_numpy(rows).to(DEV)
    # row tiles of the sampled rows: codes and scales
    rq, ri = OB.quantize_blockwise_rows(_np(a[rt]))
    assert np.array_equal(qa[rt].cpu().numpy(), rq) and np.array_equal(sa[:, rt].cpu().numpy(), ri)
    a_deq = OB.dequant_rows(rq, ri)
    # weight slabs (128 output rows of one expert, every k tile) for sampled columns
    ncols = np.array(sorted(set(rng.integers(0, N, size=6).tolist() + [N - 1])))
    w_deq = {}
    for e in np.unique(grp):
        for nb in sorted(set(int(n) // 128 for n in ncols)):
            slab = _np(w[int(e), nb * 128:(nb + 1) * 128])[None]
            q, s = OB.quantize_blockwise_weight(slab)
            assert np.array_equal(qw[int(e), nb * 128:(nb + 1) * 128].cpu().numpy(), q[0])
            assert np.array_equal(sw[int(e), nb].cpu().numpy(), s[0, 0])
            w_deq[(int(e), nb)] = OB.dequant_weight(q, s)[0]
    got = _np(out[rt][:, torch.from_numpy(ncols).to(DEV)])
    ref = np.zeros_like(got, dtype=np.float64)
    bnd = np.zeros_like(ref)
    for i, (r, e) in enumerate(zip(rows, grp)):
        wr = np.stack([w_deq[(int(e), int(n) // 128)][int(n) % 128] for n in ncols])
        ref[i] = wr @ a_deq[i]
        bnd[i] = np.abs(wr) @ np.abs(a_deq[i])
    _check_vals(got, ref, bnd, "blockwise fwd")

    # dgrad: dY row tiles along N against W^T (the same 128x128 tiles)
    kcols = np.array(sorted(set(rng.integers(0, K, size=4).tolist())))
    dq, di = OB.quantize_blockwise_rows(_np(dy[rt]))
    assert np.array_equal(qdy[rt].cpu().numpy(), dq) and np.array_equal(sdy[:, rt].cpu().numpy(), di)
    dy_deq = OB.dequant_rows(dq, di)
    got = _np(da[rt][:, torch.from_numpy(kcols).to(DEV)])
    ref = np.zeros_like(got, dtype=np.float64)
    bnd = np.zeros_like(ref)
    for e in np.unique(grp):
        sel = grp == e
        cols = []
        for k in kcols:
            kb = int(k) // 128
            slab = _np(w[int(e), :, kb * 128:(kb + 1) * 128])[None]       # [1, N, 128]
            q, s = OB.quantize_blockwise_weight(slab)
            assert np.array_equal(qwt[int(e), int(k)].cpu().numpy(), q[0][:, int(k) % 128])
            cols.append(OB.dequant_weight(q, s)[0][:, int(k) % 128])       # W[e, :, k] over N
        wt = np.stack(cols)                                               # [k, N]
        ref[sel] = dy_deq[sel] @ wt.T
        bnd[sel] = np.abs(dy_deq[sel]) @ np.abs(wt).T
    _check_vals(got, ref, bnd, "blockwise dgrad")

    # wgrad: token tiles of sampled columns (codes and scales), then a few
    # (n, k) of every expert
    nn = rng.integers(0, N, size=4)
    kk = rng.integers(0, K, size=4)
    nt, kt = torch.from_numpy(nn).to(DEV), torch.from_numpy(kk).to(DEV)
    tq_dy, ts_dy = OB.quantize_blockwise_tokens(_np(dy[:, nt]), offs_np)
    tq_a, ts_a = OB.quantize_blockwise_tokens(_np(a[:, kt]), offs_np)
    nblk = len(ts_dy)
    assert np.array_equal(qdyt[nt].cpu().numpy(), tq_dy) and np.array_equal(qat[kt].cpu().numpy(), tq_a)
    assert np.array_equal(sdyt[:nblk][:, nt].cpu().numpy(), ts_dy)
    assert np.array_equal(sat[:nblk][:, kt].cpu().numpy(), ts_a)
    dyt = OB.dequant_tokens(tq_dy, ts_dy, offs_np)      # [4, M]
    at = OB.dequant_tokens(tq_a, ts_a, offs_np)
    for e in range(E):
        s0, s1 = int(starts[e]), int(ends[e])
        got = _np(dw[e][nt][:, kt])
        if s1 == s0:
            assert np.all(got == 0)
            continue
        ref = dyt[:, s0:s1] @ at[:, s0:s1].T
        _check_vals(got, ref, np.abs(dyt[:, s0:s1]) @ np.abs(at[:, s0:s1]).T, f"blockwise wgrad e={e}")
