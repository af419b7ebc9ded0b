"""GPU parity of token routing (permute into 32-padded expert groups, weighted
unpermute) against the CPU oracle, bit-exact; and a routed MXFP8 layer end to
end (route -> dual quantization -> grouped GEMM -> combine)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import grouped_mm as OG, quant as OQ, routing as RT

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def F():
    from mxfp8_moe_quantization_gb300 import build as B
    B.build()
    import mxfp8_moe_quantization_gb300 as m
    return m


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


def _topk(T, k, E, seed, skew=0.0, dup=False):
    rng = np.random.default_rng(seed)
    p = np.arange(1, E + 1, dtype=np.float64) ** -skew
    p /= p.sum()
    idx = np.stack([rng.choice(E, size=k, replace=dup, p=p) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    return idx, w


def _np(t):
    return t.float().cpu().numpy()


@pytest.mark.parametrize("T,k,E,H,dup", [(300, 2, 8, 64, False), (1100, 3, 5, 40, True), (77, 1, 1, 8, False)])
def test_permute_parity(F, T, k, E, H, dup):
    x = _bf16((T, H), T + 1)
    idx, w = _topk(T, k, E, T, 1.1, dup)
    a, offs, row_of = F.fp8moe_route_permute(x.to(DEV), torch.from_numpy(idx).to(DEV), E)
    ra, roffs, rrow = RT.route_permute(_np(x), idx, E)
    assert np.array_equal(offs.cpu().numpy(), roffs)
    assert np.array_equal(row_of.cpu().numpy(), rrow)
    assert np.array_equal(_np(a), ra)
    # weighted
    aw, _, _ = F.fp8moe_route_permute(x.to(DEV), torch.from_numpy(idx).to(DEV), E, torch.from_numpy(w).to(DEV))
    raw, _, _ = RT.route_permute(_np(x), idx, E, w)
    assert np.array_equal(_np(aw), raw)
    assert F.fp8moe_get_device_status() == 0


@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("k,N", [(3, 96), (1, 2056), (2, 1032), (8, 520), (11, 264)])
def test_unpermute_parity(F, weighted, k, N):
    """Every shape of the combine kernel (source rows loaded 1, 2, 4 or 8 at a
    time; k = 11 takes a second group) and ragged column chunk counts."""
    T, E = 500, 13
    idx, w = _topk(T, k, E, 9 + k)
    _, _, rrow = RT.route_permute(np.zeros((T, 8), np.float32), idx, E)
    y = _bf16((RT.route_rows(T, k, E), N), 10)
    out = F.fp8moe_route_unpermute(y.to(DEV), torch.from_numpy(rrow).to(DEV),
                                   torch.from_numpy(w).to(DEV) if weighted else None)
    ref = RT.route_unpermute(_np(y), rrow, w if weighted else None)
    assert np.array_equal(_np(out), ref)


@pytest.mark.parametrize("name", ["scout", "dsv3"])
def test_permute_model_shapes(F, name):
    """Routing of the layer shapes the bench times (Scout top-1 over 16,
    hidden 5120; DeepSeek-V3 top-8 over 256 with a Zipf skew, hidden 7168):
    offsets and rows exact, sampled data rows bit for bit."""
    wl = W.get_workload(name)
    T, E = wl.tokens, wl.E
    k = 1 if name == "scout" else 8
    H = wl.K
    idx, w = _topk(T, k, E, 3, 0.0 if name == "scout" else 1.2)
    x = _bf16((T, H), 4)
    a, offs, row_of = F.fp8moe_route_permute(x.to(DEV), torch.from_numpy(idx).to(DEV), E)
    ra, roffs, rrow = RT.route_permute(_np(x), idx, E)
    assert np.array_equal(offs.cpu().numpy(), roffs)
    assert np.array_equal(row_of.cpu().numpy(), rrow)
    rows = np.random.default_rng(5).integers(0, a.shape[0], size=200)
    assert np.array_equal(_np(a[torch.from_numpy(rows).to(DEV)]), ra[rows])
    assert F.fp8moe_get_device_status() == 0


def test_roundtrip_and_empty(F):
    T, k, E, H = 256, 2, 6, 32
    idx, _ = _topk(T, k, E, 12)
    x = _bf16((T, H), 13)
    a, offs, row_of = F.fp8moe_route_permute(x.to(DEV), torch.from_numpy(idx).to(DEV), E)
    half = torch.full((T, k), 0.5, dtype=torch.float32, device=DEV)
    back = F.fp8moe_route_unpermute(a, row_of, half)
    assert torch.equal(back.cpu(), x)
    # no tokens: every group empty, the last one holds the (zero) slack
    xe = torch.zeros(0, H, dtype=torch.bfloat16, device=DEV)
    ie = torch.zeros(0, k, dtype=torch.int32, device=DEV)
    ae, oe, _ = F.fp8moe_route_permute(xe, ie, E)
    assert oe.cpu().tolist() == [0] * (E - 1) + [RT.route_rows(0, k, E)]
    assert torch.count_nonzero(ae).item() == 0


def test_invalid_expert_ids(F):
    T, k, E, H = 64, 2, 4, 16
    idx, _ = _topk(T, k, E, 14)
    idx[5, 1] = 7          # out of range
    idx[9, 0] = -1
    x = _bf16((T, H), 15)
    _, _, row_of = F.fp8moe_route_permute(x.to(DEV), torch.from_numpy(idx).to(DEV), E)
    assert F.fp8moe_get_device_status() == 5
    r = row_of.cpu().numpy()
    assert r[5, 1] == -1 and r[9, 0] == -1
    assert F.fp8moe_get_device_status() == 0


def test_routed_mxfp8_layer_end_to_end(F):
    """route -> dual MXFP8 quantization with the routing offsets -> grouped
    GEMM forward -> weighted combine, against the oracle chain."""
    T, k, E, K, N = 384, 2, 6, 256, 512
    idx, w = _topk(T, k, E, 21, 1.0)
    x = _bf16((T, K), 22)
    wt = _bf16((E, N, K), 23, 0.05)
    d_idx, d_w = torch.from_numpy(idx).to(DEV), torch.from_numpy(w).to(DEV)
    a, offs, row_of = F.fp8moe_route_permute(x.to(DEV), d_idx, E)
    qa, sa, _, _ = F.fp8moe_mxfp8_quantize_dual(a, offs, F.GROUP_ROWS, F.GROUP_COLS)
    qw, sw, _, _ = F.fp8moe_mxfp8_quantize_dual(wt.to(DEV), None, F.NO_GROUPS, F.NO_GROUPS, dim1=False)
    y = F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, qa, sa, qw, sw, offs)
    out = F.fp8moe_route_unpermute(y, row_of, d_w)
    assert F.fp8moe_get_device_status() == 0
    # oracle chain
    ra, roffs, rrow = RT.route_permute(_np(x), idx, E)
    qa_r, sa_r = OQ.mxfp8_quantize_dim0(ra)
    qw_r, sw_r = OQ.mxfp8_quantize_dim0(_np(wt))
    ref_y, bound_y = OG.grouped_mm_fwd(OQ.dequant_mx(qa_r, sa_r), OQ.dequant_mx(qw_r, sw_r), roffs)
    ref = sum(w[:, j:j + 1].astype(np.float64) * ref_y[rrow[:, j]] for j in range(k))
    bound = sum(w[:, j:j + 1].astype(np.float64) * (8e-3 * np.abs(ref_y[rrow[:, j]]) + 1e-3 * bound_y[rrow[:, j]]
                                                    + 2.0 ** -8 * np.abs(ref_y[rrow[:, j]])) for j in range(k))
    got = _np(out)
    assert np.all(np.abs(got - ref) <= bound + 2.0 ** -8 * np.abs(ref))


@pytest.mark.parametrize("name", ["scout", "dsv3"])
def test_unpermute_model_shapes(F, name):
    """The weighted combine at the layer shapes the bench times (Scout top-1
    over 16 experts, hidden 5120; DeepSeek-V3 top-8 over 256, hidden 7168):
    sampled tokens bit for bit against the oracle, which recombines them
    from just the expert-output rows they read."""
    wl = W.get_workload(name)
    T, E, N = wl.tokens, wl.E, wl.K
    k = 1 if name == "scout" else 8
    idx, w = _topk(T, k, E, 21, 0.0 if name == "scout" else 1.2)
    _, _, rrow = RT.route_permute(np.zeros((T, 8), np.float32), idx, E)
    g = torch.Generator(device=DEV).manual_seed(22)
    y = torch.randn(RT.route_rows(T, k, E), N, device=DEV, generator=g).to(torch.bfloat16)
    out = F.fp8moe_route_unpermute(y, torch.from_numpy(rrow).to(DEV), torch.from_numpy(w).to(DEV))
    torch.cuda.synchronize()
    assert F.fp8moe_get_device_status() == 0
    tok = np.unique(np.concatenate([[0, T - 1], np.random.default_rng(23).integers(0, T, size=62)]))
    sub = rrow[tok]
    need = np.unique(sub)
    local = np.searchsorted(need, sub)
    ysub = _np(y[torch.from_numpy(need).to(DEV)])
    ref = RT.route_unpermute(ysub, local, w[tok])
    assert np.array_equal(_np(out[torch.from_numpy(tok).to(DEV)]), ref)
