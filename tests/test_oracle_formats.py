"""Pins for the oracle's FP8 / e8m0 formats (CPU only).

Each check compares the oracle with something other than itself: constants
the pages print, torch's own CPU FP8 casts (for in-range values, where
saturation plays no role), an argmin over the whole code table, and an
integer bit-field computation of floor(log2).
"""
import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_constants.txt")


def _page_constants():
    out = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = line.split("|")[0].split()
        out[key] = val
    return out


def test_page_constants():
    pc = _page_constants()
    assert F.FP8_MAX[F.FNUZ] == float(pc["e4m3fnuz_max"])
    tab = F.decode_table(F.FNUZ)
    assert np.nanmax(tab) == 240.0
    # FNUZ: no infinities; the single NaN is not a "NaN encoding" of a value
    assert not np.isinf(tab).any()
    assert int(np.isnan(tab).sum()) == 1 and np.isnan(tab[0x80])
    assert int(pc["mx_block_elements"]) == 32


def test_e4m3fn_table_against_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    for kind, dt in [(F.FN, torch.float8_e4m3fn), (F.FNUZ, torch.float8_e4m3fnuz)]:
        ref = codes.view(dt).to(torch.float64).numpy()
        ours = F.decode_table(kind)
        fin = np.isfinite(ref)
        assert np.array_equal(np.isnan(ours), np.isnan(ref))
        assert np.array_equal(ours[fin], ref[fin])
    assert np.nanmax(F.decode_table(F.FN)) == 448.0
    assert np.nanmin(np.abs(F.decode_table(F.FN))[1:0x7F]) == 2.0 ** -9
    assert np.nanmin(np.abs(F.decode_table(F.FNUZ))[1:0x7F]) == 2.0 ** -10


@pytest.mark.parametrize("kind", [F.FN, F.FNUZ])
def test_roundtrip_all_codes(kind):
    tab = F.decode_table(kind)
    for c in range(256):
        if np.isnan(tab[c]):
            continue
        got = int(F.encode(np.array([tab[c]]), kind)[0])
        if kind == F.FNUZ and tab[c] == 0:
            assert got == 0
        else:
            assert got == c, (kind, hex(c), hex(got))


def _all_bf16_as_f32():
    bits = np.arange(65536, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    return v[np.isfinite(v)]


@pytest.mark.parametrize("kind,dt", [(F.FN, torch.float8_e4m3fn), (F.FNUZ, torch.float8_e4m3fnuz)])
def test_encode_matches_torch_in_range(kind, dt):
    """In range, RNE encoding must agree with torch's CPU cast bit for bit."""
    rng = np.random.default_rng(7)
    vmax = F.FP8_MAX[kind]
    v_bf16 = _all_bf16_as_f32()
    v_rand = (rng.standard_normal(200000) * rng.choice([1e-3, 1.0, 30.0, 200.0], 200000)).astype(np.float32)
    tab = F.decode_table(kind)
    fin = tab[np.isfinite(tab)]
    mids = ((fin[:, None] + fin[None, :]) / 2).ravel().astype(np.float32)   # tie points
    v = np.concatenate([v_bf16, v_rand, mids, np.float32([0.0, -0.0])])
    v = v[np.abs(v) <= vmax]
    ref = torch.from_numpy(v).to(dt).view(torch.uint8).numpy()
    ours = F.encode(v, kind)
    assert np.array_equal(ref, ours)


@pytest.mark.parametrize("kind", [F.FN, F.FNUZ])
def test_encode_is_nearest_even_by_argmin(kind):
    """Brute force: the code minimises |v - value|; ties go to the even code."""
    tab = F.decode_table(kind)
    codes = np.array([c for c in range(256) if np.isfinite(tab[c])])
    vals = tab[codes]
    rng = np.random.default_rng(3)
    vmax = F.FP8_MAX[kind]
    v = np.concatenate([rng.uniform(-vmax, vmax, 3000), rng.uniform(-0.01, 0.01, 2000),
                        ((vals[:, None] + vals[None, :]) / 2).ravel()[::7]])
    got = F.encode(v, kind)
    for x, c in zip(v, got):
        d = np.abs(vals - x)
        best = codes[d == d.min()]
        bestv = tab[best]
        # all minimisers have equal value up to the sign of zero
        if len(set(np.abs(bestv))) > 1:
            best = best[(best & 1) == 0]
        if x == 0 or np.all(tab[best] == 0):
            assert tab[c] == 0
        else:
            assert tab[c] in set(tab[best]), (x, hex(c), [hex(b) for b in best])


def test_saturation_and_zero_sign():
    assert F.encode(np.array([1e30, -1e30, 449.0, 480.0]), F.FN).tolist() == [0x7E, 0xFE, 0x7E, 0x7E]
    assert F.encode(np.array([1e30, -1e30, 241.0, 448.0]), F.FNUZ).tolist() == [0x7F, 0xFF, 0x7F, 0x7F]
    assert F.encode(np.array([-0.0, -1e-30, 0.0]), F.FN).tolist() == [0x80, 0x80, 0x00]
    assert F.encode(np.array([-0.0, -1e-30, 0.0]), F.FNUZ).tolist() == [0, 0, 0]
    # the fnuz NaN code is never produced from finite input
    rng = np.random.default_rng(1)
    v = rng.standard_normal(100000) * 100
    assert not np.any(F.encode(v, F.FNUZ) == 0x80)


def _floor_log2_bits(v32: np.ndarray) -> np.ndarray:
    """floor(log2|v|) for finite nonzero fp32 values, from the bit fields."""
    b = np.abs(v32).view(np.uint32).astype(np.int64)
    ef = b >> 23
    man = b & 0x7FFFFF
    out = ef - 127
    sub = ef == 0
    # subnormal: value = man * 2^-149 -> floor(log2) = msb(man) - 149
    msb = np.zeros_like(man)
    m = man.copy()
    for _ in range(23):
        nz = m > 1
        msb += nz
        m = np.where(nz, m >> 1, m)
    return np.where(sub, msb - 149, out)


def test_e8m0_exhaustive_bf16():
    v = _all_bf16_as_f32()
    v = np.abs(v)
    got = F.e8m0_from_amax(v).astype(np.int64)
    nz = v > 0
    E = _floor_log2_bits(v[nz].astype(np.float32))
    want = np.clip(E - 8, -127, 127) + 127
    assert np.array_equal(got[nz], want)
    assert np.all(got[~nz] == 0)
    assert got.max() <= 254
    # closed forms
    assert F.e8m0_from_amax(np.array([448.0, 1.0, 2.0 ** 20, 511.0, 512.0])).tolist() == \
        [127, 119, 139, 127, 128]


def test_e8m0_block_max_lands_in_256_448():
    """After division by 2^e the block maximum encodes to [256, 448]."""
    v = _all_bf16_as_f32()
    v = np.abs(v[(v != 0)])
    b = F.e8m0_from_amax(v).astype(np.int64)
    e = b - 127
    scaled = np.abs(v.astype(np.float64)) * np.ldexp(1.0, (-e).astype(np.int32))
    unclamped = (b > 0)
    q = F.decode(F.encode(scaled[unclamped], F.FN))
    assert q.min() >= 256 and q.max() <= 448
