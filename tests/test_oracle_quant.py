"""Pins for the oracle's quantizers, swizzle and grouped GEMM (CPU only)."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import quant as Q
from oracle import swizzle as S
from oracle import grouped_mm as G


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def _rand(shape, seed, scale=1.0):
    return _bf16(np.random.default_rng(seed).standard_normal(shape) * scale)


# ----------------------------------------------------------------------------
# rowwise / colwise
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("kind", [F.FN, F.FNUZ])
def test_rowwise_amax_maps_to_max(kind):
    x = _rand((64, 300), 1, 3.0)
    x[5] = 0.0
    q, inv = Q.quantize_rowwise(x, kind)
    top = 0x7E if kind == F.FN else 0x7F
    for r in range(64):
        if r == 5:
            assert np.all(q[r] == 0)
            continue
        i = np.argmax(np.abs(x[r]))
        assert q[r, i] == (top | (0x80 if x[r, i] < 0 else 0))
        assert np.all((q[r] & 0x7F) <= top)
    if kind == F.FNUZ:
        assert not np.any(q == 0x80)


@pytest.mark.parametrize("kind", [F.FN, F.FNUZ])
def test_rowwise_representable_rows_roundtrip(kind):
    """x = code values * 2^j whose maximum is fp8_max * 2^j quantizes to the codes."""
    rng = np.random.default_rng(2)
    tab = F.decode_table(kind)
    fin = [c for c in range(256) if np.isfinite(tab[c]) and not (kind == F.FNUZ and c == 0)]
    top = 0x7E if kind == F.FN else 0x7F
    for j in [-5, 0, 3]:
        codes = rng.choice(fin, size=(8, 64)).astype(np.uint8)
        codes[:, 0] = top
        x = (tab[codes] * 2.0 ** j).astype(np.float32)
        q, inv = Q.quantize_rowwise(x, kind)
        assert np.array_equal(q, codes)
        assert np.all(inv == np.float32(2.0 ** j))


def test_rowwise_error_bound():
    """|dequant - x| <= half an e4m3 step (relative 2^-4, or 2^-10 absolute in
    the scaled domain) -- fails if the scale is dropped or inverted."""
    x = _rand((32, 512), 3, 5.0)
    q, inv = Q.quantize_rowwise(x, F.FN)
    deq = Q.dequant_rows(q, inv)
    scaled_err = np.abs(deq - x) / inv[:, None]
    bound = np.maximum(np.abs(x) / inv[:, None] * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6)
    assert np.all(scaled_err <= bound)


@pytest.mark.parametrize("kind", [F.FN, F.FNUZ])
def test_tensorwise_amax_and_nearest_code(kind):
    """The element of largest magnitude encodes to +-max; every code is the
    nearest entry of the code table to x * s (ties to the even code),
    checked by brute force over all 256 codes."""
    x = _rand((37, 53), 11, 2.5)
    x[3, 7] = -9.5                                   # the tensor's maximum
    q, inv = Q.quantize_tensorwise(x, kind)
    top = 0x7E if kind == F.FN else 0x7F
    assert q[3, 7] == (top | 0x80)
    s = np.float32(F.FP8_MAX[kind]) / np.float32(9.5)
    assert inv == np.float32(np.float32(1.0) / s)
    codes = np.arange(256)
    vals = F.decode(codes.astype(np.uint8), kind)
    finite = np.isfinite(vals)
    if kind == F.FNUZ:
        finite &= codes != 0x80
    for v, c in zip((x * s).ravel()[:400], q.ravel()[:400]):
        d = np.abs(vals[finite] - np.float64(v))
        best = codes[finite][d == d.min()]
        if len(best) > 1:       # a tie: the even mantissa
            best = best[(best & 1) == 0]
        if best[0] & 0x7F == 0 and kind == F.FN:
            assert c & 0x7F == 0
        else:
            assert c == best[0] or (c & 0x7F) == (best[0] & 0x7F) == 0


@pytest.mark.parametrize("kind", [F.FN, F.FNUZ])
def test_tensorwise_representable_roundtrip_and_zero(kind):
    """A tensor of codes times 2^j whose maximum is the largest code comes
    back exactly, with inv = 2^j; an all-zero tensor gives zero codes and
    inv = 1 / (max / 1e-12)."""
    rng = np.random.default_rng(12)
    top = 0x7E if kind == F.FN else 0x7F
    codes = rng.integers(0, top + 1, size=(16, 24)).astype(np.uint8)
    codes |= (rng.integers(0, 2, size=codes.shape) * 0x80).astype(np.uint8)
    if kind == F.FNUZ:
        codes[codes == 0x80] = 0
    codes[0, 0] = top
    j = -3
    x = F.decode(codes, kind) * 2.0 ** j
    q, inv = Q.quantize_tensorwise(x.astype(np.float32), kind)
    assert np.array_equal(q & 0x7F, codes & 0x7F)
    assert np.array_equal(q[(codes & 0x7F) != 0], codes[(codes & 0x7F) != 0])
    assert inv == np.float32(2.0 ** j)
    z = np.zeros((4, 5), np.float32)
    qz, invz = Q.quantize_tensorwise(z, kind)
    assert np.all(qz == 0)
    assert invz == np.float32(np.float32(1.0) / (np.float32(F.FP8_MAX[kind]) / np.float32(1e-12)))


def test_colwise_3d_is_rowwise_of_transpose():
    x = _rand((3, 40, 24), 4)
    qt, inv = Q.quantize_colwise_3d(x, F.FN, transpose_out=True)
    qn, inv2 = Q.quantize_colwise_3d(x, F.FN, transpose_out=False)
    assert qt.shape == (3, 24, 40) and np.array_equal(inv, inv2)
    for e in range(3):
        qr, ir = Q.quantize_rowwise(x[e].T.copy(), F.FN)
        assert np.array_equal(qt[e], qr) and np.array_equal(inv[e], ir)
        assert np.array_equal(qn[e], qr.T)


def test_colwise_jagged_layout_and_empty_group():
    x = _rand((100, 16), 5)
    offs = np.array([30, 30, 77, 100], np.int32)       # group 1 empty
    qt, inv = Q.quantize_colwise_jagged(x, offs, F.FN, transpose_out=True)
    qn, inv2 = Q.quantize_colwise_jagged(x, offs, F.FN, transpose_out=False)
    assert np.array_equal(inv, inv2)
    W = Q.jagged_t_cols(100, 4)
    assert qt.shape == (16, W) and W % 16 == 0
    starts = [0, 30, 30, 77]
    sizes = [30, 0, 47, 23]
    P = [0, 32, 32, 96]
    assert list(Q.padded_starts(offs, 32)) == P
    used = np.zeros(W, bool)
    for e in range(4):
        seg = x[starts[e]:starts[e] + sizes[e]]
        if sizes[e]:
            qr, ir = Q.quantize_rowwise(seg.T.copy(), F.FN)
            assert np.array_equal(qt[:, P[e]:P[e] + sizes[e]], qr)
            assert np.array_equal(inv[e], ir)
            assert np.array_equal(qn[starts[e]:starts[e] + sizes[e]], qr.T)
        used[P[e]:P[e] + sizes[e]] = True
    assert np.all(qt[:, ~used] == 0)
    assert np.all(inv[1] == np.float32(1.0) / (np.float32(448.0) / np.float32(1e-12)))


# ----------------------------------------------------------------------------
# MXFP8
# ----------------------------------------------------------------------------

def test_mx_dim0_against_torch_cast():
    """In range, q must equal torch's RNE cast of x * 2^-e; the top of the
    range [448, 512) saturates to 448."""
    x = _rand((16, 256), 6, 2.0)
    x[3, :32] = 0.0
    x[4, 32:64] = 1e-30
    q, sb = Q.mxfp8_quantize_dim0(x)
    assert sb.shape == (16, 8) and sb[3, 0] == 0
    e = sb.astype(np.int64) - 127
    y = x.reshape(16, 8, 32).astype(np.float64) * np.ldexp(1.0, (-e).astype(np.int32))[..., None]
    y = y.reshape(16, 256)
    inr = np.abs(y) <= 448
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q[inr], ref[inr])
    assert np.all((q[~inr] & 0x7F) == 0x7E)


def test_mx_exact_reconstruction():
    """Values that are e4m3 codes times the block's 2^e come back exactly."""
    rng = np.random.default_rng(8)
    tab = F.decode_table(F.FN)
    fin = np.array([c for c in range(256) if np.isfinite(tab[c])])
    codes = rng.choice(fin, size=(4, 64)).astype(np.uint8)
    codes[:, 0] = 0x78   # 256: block amax in [256, 512) keeps e = j
    codes[:, 32] = 0x78
    for j in [-20, 0, 7]:
        x = tab[codes] * 2.0 ** j
        x[:, 1:32][np.abs(x[:, 1:32]) > 256 * 2.0 ** j] = 0
        x[:, 33:][np.abs(x[:, 33:]) > 256 * 2.0 ** j] = 0
        q, sb = Q.mxfp8_quantize_dim0(x)
        assert np.all(sb == j + 127)
        assert np.array_equal(Q.dequant_mx(q, sb), x)


def test_mx_dim1_equals_dim0_of_transpose():
    x = _rand((2, 96, 64), 9, 4.0)
    qt, st = Q.mxfp8_quantize_dim1(x)
    assert qt.shape == (2, 64, 96) and st.shape == (2, 64, 3)
    for b in range(2):
        q0, s0 = Q.mxfp8_quantize_dim0(x[b].T.copy())
        assert np.array_equal(qt[b], q0) and np.array_equal(st[b], s0)


# ----------------------------------------------------------------------------
# swizzle
# ----------------------------------------------------------------------------

def test_swizzle_documented_positions():
    s = np.zeros((128, 4), np.uint8)
    marks = {(0, 0): 0, (0, 1): 1, (1, 0): 16, (32, 0): 4, (64, 2): 10, (96, 3): 15, (127, 3): 511}
    for i, (rc, _) in enumerate(marks.items()):
        s[rc] = i + 1
    out = S.swizzle(s)
    for i, (rc, off) in enumerate(marks.items()):
        assert out[off] == i + 1


@pytest.mark.parametrize("R,Cs", [(128, 4), (200, 7), (1, 1), (300, 12)])
def test_swizzle_bijection_and_padding(R, Cs):
    rng = np.random.default_rng(R * 31 + Cs)
    s = rng.integers(1, 256, size=(R, Cs)).astype(np.uint8)
    out = S.swizzle(s)
    Rp, Cp = S.swizzled_shape(R, Cs)
    assert out.size == Rp * Cp
    back = S.unswizzle(out, Rp, Cp)
    assert np.array_equal(back[:R, :Cs], s)
    assert np.all(back[R:] == 0) and np.all(back[:, Cs:] == 0)
    offs = S.tile_offset(np.arange(Rp)[:, None], np.arange(Cp)[None, :], Cp).ravel()
    assert np.array_equal(np.sort(offs), np.arange(Rp * Cp))


def test_swizzle_grouped_rows():
    rng = np.random.default_rng(11)
    s = rng.integers(1, 256, size=(300, 6)).astype(np.uint8)
    offs = np.array([100, 100, 260, 300], np.int32)
    out = S.swizzle(s, offs, S.GROUP_ROWS)
    Rp, Cp = S.swizzled_shape(300, 6, 4, S.GROUP_ROWS)
    back = S.unswizzle(out, Rp, Cp)
    starts = [0, 100, 100, 260]
    P = [0, 128, 128, 384]
    used = np.zeros(Rp, bool)
    for e in range(4):
        g = offs[e] - starts[e]
        assert np.array_equal(back[P[e]:P[e] + g, :6], s[starts[e]:offs[e]])
        used[P[e]:P[e] + g] = True
    assert np.all(back[~used] == 0)


def test_swizzle_grouped_cols():
    rng = np.random.default_rng(12)
    Cs = 10                                   # 320 contracting elements
    s = rng.integers(1, 256, size=(130, Cs)).astype(np.uint8)
    offs = np.array([64, 64, 320], np.int32)  # groups of 2, 0, 8 scale columns
    out = S.swizzle(s, offs, S.GROUP_COLS)
    Rp, Cp = S.swizzled_shape(130, Cs, 3, S.GROUP_COLS)
    back = S.unswizzle(out, Rp, Cp)
    assert np.array_equal(back[:130, 0:2], s[:, 0:2])
    assert np.array_equal(back[:130, 4:12], s[:, 2:10])
    mask = np.zeros((Rp, Cp), bool)
    mask[:130, 0:2] = True
    mask[:130, 4:12] = True
    assert np.all(back[~mask] == 0)


# ----------------------------------------------------------------------------
# grouped GEMM
# ----------------------------------------------------------------------------

def test_grouped_mm_brute_force():
    rng = np.random.default_rng(13)
    a = rng.standard_normal((12, 5))
    w = rng.standard_normal((3, 4, 5))
    offs = np.array([5, 5, 12])
    out, bound = G.grouped_mm_fwd(a, w, offs)
    for e, (s, t) in enumerate([(0, 5), (5, 5), (5, 12)]):
        if t > s:
            assert np.allclose(out[s:t], G.brute_force_mm(a[s:t], w[e]), rtol=1e-14, atol=1e-14)
            assert np.allclose(bound[s:t], G.brute_force_mm(np.abs(a[s:t]), np.abs(w[e])))
    # E = 1 is a plain dense GEMM
    d, _ = G.grouped_mm_fwd(a, w[:1], np.array([12]))
    assert np.allclose(d, G.brute_force_mm(a, w[0]))
    with pytest.raises(ValueError):
        G.grouped_mm_fwd(a, w, np.array([5, 5, 11]))


def test_three_gemms_are_adjoint():
    """<fwd(A,W), Gy> = <A, dgrad(Gy, W^T)> = sum_e <W_e, wgrad(Gy^T, A^T)_e>.

    Ties the three definitions together: a transposed operand or a wrong
    group slice in any of them breaks the identity.
    """
    rng = np.random.default_rng(14)
    M, K, N = 40, 6, 7
    offs = np.array([10, 10, 33, 40])
    a = rng.standard_normal((M, K))
    w = rng.standard_normal((4, N, K))
    gy = rng.standard_normal((M, N))
    y, _ = G.grouped_mm_fwd(a, w, offs)
    da, _ = G.grouped_mm_dgrad(gy, np.transpose(w, (0, 2, 1)), offs)
    dw, _ = G.grouped_mm_wgrad(gy.T, a.T, offs)
    l0 = np.sum(y * gy)
    assert np.isclose(l0, np.sum(a * da), rtol=1e-12)
    assert np.isclose(l0, np.sum(w * dw), rtol=1e-12)
    assert np.all(dw[1] == 0)
    # summing wgrad over groups is the dense product
    assert np.allclose(dw.sum(0), gy.T @ a)
