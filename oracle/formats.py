"""FP8 number formats, written out from their definitions (CPU oracle).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this file.

* e4m3fn  ("the NVIDIA format"): 1 sign, 4 exponent bits (bias 7), 3 mantissa
  bits; exponent field 0 is subnormal (m/8 * 2^-6); code S.1111.111 is NaN;
  there is no infinity; largest finite magnitude 1.75 * 2^8 = 448.
  The pages contrast it with FNUZ and stress that using the other format's
  maximum silently clips ("FP8-обучение на AMD", section "Тихая порча
  градиентов: проблема формата FNUZ").
* e4m3fnuz (AMD Instinct): bias 8, exponent field 0 is subnormal
  (m/8 * 2^-7), the only NaN is 0x80 (negative zero's code), no infinity,
  unsigned zero, largest finite magnitude 1.875 * 2^7 = 240.  The pages give
  max 240 and "no NaN/Inf encodings" ("FP8 training on AMD GPUs with
  TorchTitan and TorchAO" summary, section details, e4m3fnuz property table;
  glossary entry FNUZ).
* e8m0: an unsigned biased power-of-two exponent, value 2^(byte-127), one
  per 1x32 block of e4m3 data ("Accelerating Llama4 Scout training with
  TorchAO MXFP8 MoE primitives", MXFP8 data / scale-factor layout diagram).

Encoding rule (the pages give none; the plainest reading, also the one the
spec for this library fixes): round to nearest, ties to even, saturating to
+-max.  It is implemented here as a search for the nearest representable
value among the decoded code table -- deliberately not by bit manipulation --
so that it shares no method with the GPU path.

Readings where the pages are silent:
* e4m3fn keeps the sign of zero: a negative value that rounds to zero gives
  0x80.
* e4m3fnuz has an unsigned zero: anything that rounds to zero gives 0x00,
  and 0x80 is never produced.
* NaN/Inf inputs are outside the workloads; NaN maps to the format's NaN
  code (0x7F fn, 0x80 fnuz), +-Inf saturates.  Tests never feed them.
"""
from __future__ import annotations

import numpy as np

FN = "e4m3fn"
FNUZ = "e4m3fnuz"
FP8_MAX = {FN: 448.0, FNUZ: 240.0}


def decode_table(kind: str) -> np.ndarray:
    """Value of each of the 256 codes (float64; NaN for NaN codes)."""
    out = np.empty(256, dtype=np.float64)
    bias, sub_exp = (7, -6) if kind == FN else (8, -7)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if kind == FN and e == 15 and m == 7:
            out[c] = np.nan
            continue
        if kind == FNUZ and c == 0x80:
            out[c] = np.nan
            continue
        if e == 0:
            mag = (m / 8.0) * 2.0 ** sub_exp
        else:
            mag = (1.0 + m / 8.0) * 2.0 ** (e - bias)
        out[c] = s * mag
    return out


def _positive_codes(kind: str):
    """Non-negative finite magnitudes in increasing order, with their codes."""
    tab = decode_table(kind)
    codes = np.array([c for c in range(0x80) if np.isfinite(tab[c])], dtype=np.int64)
    mags = tab[codes]
    assert np.all(np.diff(mags) > 0)
    return mags, codes


_POS = {FN: _positive_codes(FN), FNUZ: _positive_codes(FNUZ)}


def decode(codes: np.ndarray, kind: str = FN) -> np.ndarray:
    return decode_table(kind)[np.asarray(codes, dtype=np.uint8)]


def encode(v, kind: str = FN) -> np.ndarray:
    """Nearest e4m3 code (ties to even code), saturating at +-max.

    ``v`` is any float array; its values are taken exactly (float64).
    """
    v = np.asarray(v)
    x = v.astype(np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    mags, codes = _POS[kind]
    vmax = mags[-1]
    nan_in = np.isnan(a)
    a = np.minimum(np.where(nan_in, 0.0, a), vmax)          # saturate
    i = np.searchsorted(mags, a, side="right") - 1         # mags[i] <= a
    i = np.clip(i, 0, len(mags) - 1)
    j = np.minimum(i + 1, len(mags) - 1)
    lo, hi = mags[i], mags[j]
    mid = (lo + hi) / 2.0                                  # exact in float64
    up = a > mid
    tie = (a == mid) & (j != i)
    # on a tie take the code whose mantissa LSB is 0 (the even code)
    up = np.where(tie, (codes[j] & 1) == 0, up)
    mag_code = np.where(up, codes[j], codes[i])
    if kind == FN:
        out = mag_code | np.where(neg, 0x80, 0)
        out = np.where(nan_in, 0x7F, out)
    else:
        out = np.where((mag_code != 0) & neg, mag_code | 0x80, mag_code)
        out = np.where(nan_in, 0x80, out)
    return out.astype(np.uint8)


def e8m0_from_amax(amax) -> np.ndarray:
    """Biased e8m0 block scale byte for a block absolute maximum.

    Rule: e = floor(log2(amax)) - 8, clamped to [-127, 127]; byte = e + 127.
    The "-8" is log2 of the largest power of two below the e4m3fn maximum
    (256 <= 448 < 512), so the block maximum lands in [256, 512) after
    division by 2^e.  ``amax == 0`` (an all-zero block) gives e = -127,
    byte 0.  0xFF (NaN) is never produced.

    floor(log2) is taken exactly with ``frexp`` (amax = f * 2^x, f in
    [0.5, 1)), so it also covers fp32 subnormals.
    """
    a = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(a)
    E = ex.astype(np.int64) - 1
    e = np.clip(E - 8, -127, 127)
    e = np.where(a == 0, -127, e)
    return (e + 127).astype(np.uint8)


def e8m0_value(byte) -> np.ndarray:
    """2^(byte - 127) as float64 (byte 255 is NaN)."""
    b = np.asarray(byte, dtype=np.int64)
    return np.where(b == 255, np.nan, np.ldexp(1.0, (b - 127).astype(np.int32)))
