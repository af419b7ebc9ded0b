"""Pins for the blockwise oracle (CPU only): every tile reduces to an already
pinned granularity (a 1 x 128 tile is a row of a 128-column matrix, a
128 x 128 tile is a whole tensor, a token tile is one expert's column set),
plus invariants and exact round trips."""
import numpy as np
import pytest
import torch

from oracle import blockwise as BW, formats as OF, quant as OQ


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def _x(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape) * scale
    x *= np.exp(rng.uniform(-4, 4, size=shape[:-1] + (1,)))      # rows of different magnitude
    return _bf16(x)


@pytest.mark.parametrize("kind", [OF.FN, OF.FNUZ])
def test_rows_are_rowwise_per_tile(kind):
    x = _x((37, 384), 1)
    x[3, 128:256] = 0.0                                          # an all-zero tile
    q, inv = BW.quantize_blockwise_rows(x, kind)
    assert q.shape == (37, 384) and inv.shape == (3, 37)
    for b in range(3):
        rq, rinv = OQ.quantize_rowwise(x[:, b * 128:(b + 1) * 128], kind)
        assert np.array_equal(q[:, b * 128:(b + 1) * 128], rq)
        assert np.array_equal(inv[b], rinv)


def test_weight_is_tensorwise_per_tile():
    w = _x((2, 256, 384), 2, 0.02)
    q, inv = BW.quantize_blockwise_weight(w)
    assert inv.shape == (2, 2, 3)
    for e in range(2):
        for nb in range(2):
            for kb in range(3):
                sl = (e, slice(nb * 128, (nb + 1) * 128), slice(kb * 128, (kb + 1) * 128))
                rq, rinv = OQ.quantize_tensorwise(w[sl], OF.FN)
                assert np.array_equal(q[sl], rq) and inv[e, nb, kb] == rinv
                # the tile's absolute maximum encodes to +-448 (0x7E / 0xFE)
                i = np.unravel_index(np.argmax(np.abs(w[sl])), (128, 128))
                assert q[sl][i] & 0x7F == 0x7E


def test_token_blocks_cut_per_group():
    offs = np.array([0, 96, 96, 416, 448, 608], np.int32)         # sizes 0, 96, 0, 320, 32, 160
    blocks = BW.token_blocks(offs)
    assert blocks == [(1, 0, 96), (3, 96, 224), (3, 224, 352), (3, 352, 416), (4, 416, 448),
                      (5, 448, 576), (5, 576, 608)]
    sizes = np.diff(np.concatenate([[0], offs]))
    assert len(blocks) == int(np.sum((sizes + 127) // 128))


def test_tokens_are_colwise_per_block():
    offs = np.array([160, 160, 448], np.int32)
    x = _x((448, 48), 3)
    qt, inv = BW.quantize_blockwise_tokens(x, offs)
    assert qt.shape == (48, 448) and inv.shape == (len(BW.token_blocks(offs)), 48)
    for i, (_, b0, b1) in enumerate(BW.token_blocks(offs)):
        rq, rinv = OQ.quantize_colwise_3d(x[None, b0:b1], OF.FN, transpose_out=True)
        assert np.array_equal(qt[:, b0:b1], rq[0]) and np.array_equal(inv[i], rinv[0])
    with pytest.raises(ValueError):
        BW.quantize_blockwise_tokens(x, np.array([100, 100, 448], np.int32))   # not a multiple of 32


def test_exact_round_trip_of_representable_tiles():
    rng = np.random.default_rng(4)
    tab = OF.decode_table(OF.FN)
    fin = tab[np.isfinite(tab)]
    # every tile holds fp8 values times 2^j with its maximum exactly 448 * 2^j
    x = rng.choice(fin, size=(64, 256))
    x[:, 0] = 448.0
    x[:, 128] = -448.0
    j = rng.integers(-20, 20, size=(64, 2))
    x = x * np.repeat(np.ldexp(1.0, j), 128, axis=1)
    x = x.astype(np.float32)
    q, inv = BW.quantize_blockwise_rows(x)
    assert np.array_equal(BW.dequant_rows(q, inv), x.astype(np.float64))
    w = (rng.choice(fin, size=(1, 128, 128)) * 2.0 ** -7).astype(np.float32)
    w[0, 5, 9] = 448.0 * 2.0 ** -7
    qw, iw = BW.quantize_blockwise_weight(w)
    assert np.array_equal(BW.dequant_weight(qw, iw), w.astype(np.float64))


def test_dequant_matches_elementwise_definition():
    x = _x((5, 256), 5)
    q, inv = BW.quantize_blockwise_rows(x)
    d = BW.dequant_rows(q, inv)
    dec = OF.decode(q, OF.FN)
    for r in range(5):
        for c in range(0, 256, 17):
            assert d[r, c] == dec[r, c] * np.float64(inv[c // 128, r])
    offs = np.array([64, 224], np.int32)
    xt = _x((224, 16), 6)
    qt, it = BW.quantize_blockwise_tokens(xt, offs)
    dt = BW.dequant_tokens(qt, it, offs)
    dect = OF.decode(qt, OF.FN)
    for i, (_, b0, b1) in enumerate(BW.token_blocks(offs)):
        assert np.array_equal(dt[:, b0:b1], dect[:, b0:b1] * it[i].astype(np.float64)[:, None])
