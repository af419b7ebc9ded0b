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
from oracle import formats as OF, quant as OQ

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


@pytest.mark.parametrize("name", ["scout", "dsv3"])
def test_mxfp8_fullsize(F, name):
    wl = W.get_workload(name)
    rng = np.random.default_rng(7)
    M, E, N, K = wl.M, wl.E, wl.N, wl.K
    offs_np = wl.offs()
    offs = torch.from_numpy(offs_np).to(DEV)
    a = W.make_activations(wl, "A", device=DEV)
    dy = W.make_activations(wl, "dY", device=DEV)
    w = W.make_weights(wl, "W1", device=DEV)
    qa, sa, qat, sat = F.fp8moe_mxfp8_quantize_dual(a, offs, F.GROUP_ROWS, F.GROUP_COLS)
    qw, sw, qwt, swt = F.fp8moe_mxfp8_quantize_dual(w, None, F.NO_GROUPS, F.NO_GROUPS)
    qdy, sdy, qdyt, sdyt = F.fp8moe_mxfp8_quantize_dual(dy, offs, F.GROUP_ROWS, F.GROUP_COLS)
    out = F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, qa, sa, qw, sw, offs)
    da = F.fp8moe_scaled_grouped_mm_dgrad(F.MXFP8, qdy, sdy, qwt, swt, offs)
    dw = F.fp8moe_scaled_grouped_mm_wgrad(F.MXFP8, qdyt, sdyt, qat, sat, offs, M)
    torch.cuda.synchronize()
    assert F.fp8moe_get_device_status() == 0

    rows = _sample_rows(offs_np, rng)
    starts, ends = OQ.group_bounds(offs_np)
    grp = np.searchsorted(ends, rows, side="right")
    # quantized codes of sampled rows (dim0) and of a column slice (dim1)
    a_rows = _np(a[torch.from_numpy(rows).to(DEV)])
    rq, _ = OQ.mxfp8_quantize_dim0(a_rows)
    assert np.array_equal(qa[torch.from_numpy(rows).to(DEV)].cpu().numpy(), rq)
    c0 = int(rng.integers(0, K // 64)) * 64
    rqt, _ = OQ.mxfp8_quantize_dim1(_np(a[:, c0:c0 + 64]))
    assert np.array_equal(qat[c0:c0 + 64].cpu().numpy(), rqt)

    # forward: sampled rows x sampled columns
    ncols = np.array(sorted(set(rng.integers(0, N, size=24).tolist() + [0, N - 1])))
    a_deq = _mx_rows(a_rows)
    got = _np(out[torch.from_numpy(rows).to(DEV)][:, torch.from_numpy(ncols).to(DEV)])
    ref = np.zeros_like(got, dtype=np.float64)
    bnd = np.zeros_like(ref)
    for e in np.unique(grp):
        sel = grp == e
        w_deq = _mx_rows(_np(w[int(e)][torch.from_numpy(ncols).to(DEV)]))
        ref[sel] = a_deq[sel] @ w_deq.T
        bnd[sel] = np.abs(a_deq[sel]) @ np.abs(w_deq).T
    _check_vals(got, ref, bnd, f"{name} fwd")

    # dgrad: sampled rows x sampled K columns (W quantized along N)
    kcols = np.array(sorted(set(rng.integers(0, K, size=16).tolist() + [K - 1])))
    dy_deq = _mx_rows(_np(dy[torch.from_numpy(rows).to(DEV)]))
    got = _np(da[torch.from_numpy(rows).to(DEV)][:, torch.from_numpy(kcols).to(DEV)])
    ref = np.zeros_like(got, dtype=np.float64)
    bnd = np.zeros_like(ref)
    for e in np.unique(grp):
        sel = grp == e
        wt_deq = _mx_cols(_np(w[int(e)][:, torch.from_numpy(kcols).to(DEV)]))   # [k, N]
        ref[sel] = dy_deq[sel] @ wt_deq.T
        bnd[sel] = np.abs(dy_deq[sel]) @ np.abs(wt_deq).T
    _check_vals(got, ref, bnd, f"{name} dgrad")

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
        _check_vals(got, dyc @ ac.T, np.abs(dyc) @ np.abs(ac).T, f"{name} wgrad e={e}")


@pytest.mark.parametrize("name", ["llama3_8b", "dsmoe_16b"])
def test_rowwise_fullsize(F, name):
    wl = W.get_workload(name)
    rng = np.random.default_rng(11)
    M, E, N, K = wl.M, wl.E, wl.N, wl.K
    offs_np = wl.offs()
    offs = torch.from_numpy(offs_np).to(DEV)
    a = W.make_activations(wl, "A", device=DEV)
    dy = W.make_activations(wl, "dY", device=DEV)
    w = W.make_weights(wl, "W1", device=DEV)
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
    _check_vals(got, ref, bnd, f"{name} fwd")

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
    _check_vals(got, ref, bnd, f"{name} dgrad")

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
        _check_vals(got, dyc @ ac.T, np.abs(dyc) @ np.abs(ac).T, f"{name} wgrad e={e}")


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
