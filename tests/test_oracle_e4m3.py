"""Pins for the oracle's E4M3 codec (CPU only).

What fixes each expected value:
  * tests/golden/e4m3_codes.txt -- values of selected codes as stated by the
    OCP 8-bit floating point specification (E4M3: bias 7, max 448, NaN at
    S.1111.111);
  * the format's closed form, checked code by code as exact rationals;
  * invariants: the 127 non-negative finite codes are strictly increasing,
    the negative half mirrors them;
  * brute force: the encoder's output is the nearest of the 253 distinct
    finite grid values, ties broken towards the even mantissa, magnitudes
    above 448 saturating -- over every BF16 bit pattern, random FP32 patterns
    and every midpoint of the grid +-1 FP32 ulp;
  * an independent library (ml_dtypes.float8_e4m3fn) on all codes and on
    in-range encodes, where it is installed.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_codes.txt")


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, val = line.split()
            rows.append((int(code, 16), val))
    return rows


def test_decode_golden_values():
    rows = _golden()
    assert len(rows) >= 20
    dec = oracle.e4m3_decode(np.array([c for c, _ in rows], np.uint8))
    for (code, val), got in zip(rows, dec):
        if val == "nan":
            assert math.isnan(got), hex(code)
            continue
        num, den = val.split("/")
        want = Fraction(int(num.replace("-", "")), int(den))
        neg = num.startswith("-")
        assert Fraction(float(abs(got))) == want, hex(code)
        assert math.copysign(1.0, got) == (-1.0 if neg else 1.0), hex(code)


def test_decode_closed_form_all_codes():
    dec = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            assert math.isnan(dec[c])
            continue
        mag = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        assert Fraction(float(abs(dec[c]))) == mag
        assert math.copysign(1.0, dec[c]) == (-1.0 if s else 1.0)


def test_decode_invariants():
    dec = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    pos = dec[:0x7F]
    assert np.all(np.diff(pos) > 0), "non-negative finite codes must increase strictly"
    assert pos[-1] == 448.0 and pos[0] == 0.0
    assert np.array_equal(dec[0x80:0xFF], -pos)
    assert np.isnan(dec[0x7F]) and np.isnan(dec[0xFF])
    assert math.copysign(1.0, dec[0x80]) == -1.0


def test_decode_matches_ml_dtypes():
    mld = pytest.importorskip("ml_dtypes")
    codes = np.arange(256, dtype=np.uint8)
    ref = codes.view(mld.float8_e4m3fn).astype(np.float64)
    dec = oracle.e4m3_decode(codes)
    fin = ~np.isnan(ref)
    assert np.array_equal(np.isnan(dec), ~fin)
    assert np.array_equal(dec[fin], ref[fin])
    assert np.array_equal(np.signbit(dec[fin]), np.signbit(ref[fin]))


@pytest.mark.parametrize("value,code", [
    (448.0, 0x7E), (464.0, 0x7E), (470.0, 0x7E), (1e9, 0x7E), (float("inf"), 0x7E),
    (-448.0, 0xFE), (-1e30, 0xFE), (float("-inf"), 0xFE),
    (2.0 ** -10, 0x00),            # tie between 0 and 2^-9 -> even (0)
    (1.5 * 2.0 ** -10, 0x01),      # above the tie -> 2^-9
    (3 * 2.0 ** -10, 0x02),        # tie between 2^-9 (odd) and 2*2^-9 (even)
    (1.0625, 0x38),                # tie between 1.0 and 1.125 -> 1.0 (even)
    (1.1875, 0x3A),                # tie between 1.125 and 1.25 -> 1.25 (even)
    (1.0, 0x38), (-1.0, 0xB8), (0.0, 0x00), (-0.0, 0x80), (-1e-30, 0x80),
    (15 * 2.0 ** -10, 0x08),       # tie between 7*2^-9 (odd) and 2^-6 (even)
    (240.0, 0x77), (248.0, 0x78),  # 248 ties 240 (odd) and 256 (even)
])
def test_encode_corner_cases(value, code):
    assert int(oracle.e4m3_encode(np.float32(value))) == code


def _brute_force_encode(v: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 value by exhaustive search over the grid; ties go
    to the code with an even mantissa; the sign is taken from v."""
    codes = np.arange(0x7F, dtype=np.uint8)                       # 0x00..0x7E
    grid = oracle.e4m3_decode(codes)                               # pinned above
    a = np.abs(v.astype(np.float64))
    out = np.empty(v.shape, np.uint8)
    for lo in range(0, v.size, 1 << 16):
        # beyond 448 the nearest grid point is 448 whatever the magnitude;
        # capping at 1024 keeps the distances exact in double
        aa = np.minimum(a[lo:lo + (1 << 16)], 1024.0)
        d = np.abs(aa[:, None] - grid[None, :])
        best = d.min(axis=1, keepdims=True)
        cand = d == best
        even = (codes & 1) == 0
        n_cand = cand.sum(axis=1)
        pick = np.where(n_cand == 1, cand.argmax(axis=1), (cand & even[None, :]).argmax(axis=1))
        out[lo:lo + aa.size] = codes[pick]
    out[np.isinf(a)] = 0x7E
    sign = np.signbit(v).astype(np.uint8) << 7
    return out | sign


def test_encode_brute_force_all_bf16_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    v = v[~np.isnan(v)]
    assert np.array_equal(oracle.e4m3_encode(v), _brute_force_encode(v))


def test_encode_brute_force_midpoints_and_random():
    grid = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (grid[1:] + grid[:-1]) / 2)  # exact in FP32
    near = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)),
                           np.nextafter(mids, np.float32(0)), grid.astype(np.float32),
                           np.array([464.0, 470.0, 480.0, 1e9], np.float32)])
    rng = np.random.default_rng(123)
    rand = (rng.integers(0, 1 << 32, size=400_000, dtype=np.uint64).astype(np.uint32)).view(np.float32)
    rand = rand[np.isfinite(rand)]
    scaled = (rng.standard_normal(200_000) * 60).astype(np.float32)
    v = np.concatenate([near, -near, rand, scaled])
    assert np.array_equal(oracle.e4m3_encode(v), _brute_force_encode(v))


def test_encode_decode_round_trip():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    back = oracle.e4m3_encode(oracle.e4m3_decode(codes).astype(np.float32))
    assert np.array_equal(back, codes)


def test_encode_matches_ml_dtypes_in_range():
    mld = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(7)
    v = np.concatenate([(rng.standard_normal(300_000) * 100).astype(np.float32),
                        (rng.standard_normal(100_000) * 1e-3).astype(np.float32)])
    v = v[np.abs(v) <= 448]
    ref = v.astype(mld.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(oracle.e4m3_encode(v), ref)
