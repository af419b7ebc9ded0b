"""Pins for the routing oracle (CPU only)."""
import numpy as np
import torch

from oracle import routing as RT


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def _case(T=37, k=3, E=6, H=16, seed=0):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    idx[idx == 4] = 2 if k < 3 else idx[idx == 4]     # leave some experts rarely used
    x = _bf16(rng.standard_normal((T, H)))
    return x, idx


def test_placement_matches_stable_sort():
    """Rows of expert e are its (t, j) pairs in (t, j) order: the same as a
    stable argsort of the flattened expert ids."""
    x, idx = _case()
    E = 6
    a, offs, row_of = RT.route_permute(x, idx, E)
    T, k = idx.shape
    flat = idx.ravel()
    order = np.argsort(flat, kind="stable")
    counts = np.bincount(flat, minlength=E)
    starts = np.concatenate([[0], np.cumsum((counts + 31) // 32 * 32)[:-1]])
    expect = np.empty(T * k, np.int64)
    pos = 0
    for e in range(E):
        for r in range(counts[e]):
            expect[order[pos]] = starts[e] + r
            pos += 1
    assert np.array_equal(row_of.ravel(), expect)
    for n in range(T * k):
        assert np.array_equal(a[expect[n]], x[n // k])


def test_offsets_and_padding():
    x, idx = _case(T=50, k=2, E=5, seed=1)
    E = 5
    a, offs, row_of = RT.route_permute(x, idx, E)
    assert np.all(offs % 32 == 0) and np.all(np.diff(offs) >= 0)
    assert offs[-1] == RT.route_rows(50, 2, 5) == a.shape[0]
    used = np.zeros(a.shape[0], bool)
    used[row_of.ravel()] = True
    assert np.all(a[~used] == 0)
    counts = np.bincount(idx.ravel(), minlength=E)
    starts = np.concatenate([[0], offs[:-1]])
    for e in range(E):
        rows = row_of[idx == e]
        assert np.all((rows >= starts[e]) & (rows < offs[e]))
        assert len(rows) == counts[e]


def test_weighted_roundtrip_is_exact():
    """Permute with weights 1/2, 1/2, then unpermute of the unweighted copies
    with the same weights returns x exactly (halving and doubling are exact)."""
    x, idx = _case(T=40, k=2, E=7, seed=2)
    w = np.full(idx.shape, 0.5, np.float32)
    a, offs, row_of = RT.route_permute(x, idx, 7)
    out = RT.route_unpermute(a, row_of, w)
    assert np.array_equal(out, x)
    aw, _, _ = RT.route_permute(x, idx, 7, w)
    assert np.array_equal(RT.route_unpermute(aw, row_of), x)


def test_bf16_rounding_matches_torch():
    v = np.random.default_rng(3).standard_normal(10000).astype(np.float32) * 7.0
    assert np.array_equal(RT._bf16_round(v), _bf16(v))


def test_unpermute_sum_close_to_float64():
    x, idx = _case(T=30, k=3, E=6, seed=4)
    rng = np.random.default_rng(5)
    y = _bf16(rng.standard_normal((RT.route_rows(30, 3, 6), 24)))
    w = rng.random(idx.shape).astype(np.float32)
    _, _, row_of = RT.route_permute(x, idx, 6)
    out = RT.route_unpermute(y, row_of, w)
    ref = sum(w[:, j:j + 1].astype(np.float64) * y[row_of[:, j]] for j in range(3))
    assert np.all(np.abs(out - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)
