"""Pins for the oracle's E4M3 codec: the format's own table (hand-derived
fixtures), a library codec (ml_dtypes) and brute-force nearest-grid search.
None of these reuses the oracle's arithmetic."""
import math

import ml_dtypes
import numpy as np
import pytest

import oracle


def _f(h):
    return float.fromhex(h)


def test_decode_fixture(golden):
    for code, value, why in golden("e4m3_decode_cases.txt"):
        got = oracle.e4m3_decode(np.array([int(code, 16)], dtype=np.uint8))[0]
        if value == "nan":
            assert math.isnan(got), why
        else:
            want = _f(value)
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, why)


def test_encode_fixture(golden):
    for value, code, why in golden("e4m3_encode_cases.txt"):
        v = np.float32(_f(value))
        assert float(v) == _f(value), "fixture value must be exact in fp32"
        got = int(oracle.e4m3_encode(np.array([v]))[0])
        assert got == int(code, 16), (value, why, hex(got))


def test_decode_all_codes_match_library():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    lib = codes.view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    nan = np.isnan(lib)
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], lib[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(lib[~nan]))


def test_grid_round_trip():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_midpoints_ties_to_even():
    # Every midpoint between adjacent non-negative grid values: the result is
    # the neighbour with an even mantissa (code LSB 0).
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))  # 0 .. 448
    for i in range(len(pos) - 1):
        mid = np.float32((pos[i] + pos[i + 1]) / 2)
        assert float(mid) == (pos[i] + pos[i + 1]) / 2  # exact in fp32
        want = i if i % 2 == 0 else i + 1
        assert oracle.e4m3_encode(np.array([mid]))[0] == want
        assert oracle.e4m3_encode(np.array([-mid]))[0] == want | 0x80
        # one fp32 ulp either side of the midpoint decides by distance
        lo = np.nextafter(mid, np.float32(0))
        hi = np.nextafter(mid, np.float32(1e9))
        assert oracle.e4m3_encode(np.array([lo]))[0] == i
        assert oracle.e4m3_encode(np.array([hi]))[0] == i + 1


def test_saturation():
    big = np.array([448, 449, 463.99, 464, 480, 1e4, 3.0e38], dtype=np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)


def test_random_values_match_library_after_clip():
    # ml_dtypes rounds float32 -> e4m3fn to nearest even but does not
    # saturate, so values are clipped to +-448 first.
    rng = np.random.default_rng(1)
    parts = [
        rng.standard_normal(200_000).astype(np.float32) * 100,
        rng.standard_normal(200_000).astype(np.float32) * 2.0 ** -8,  # subnormal range
        (rng.uniform(-1, 1, 200_000) * 500).astype(np.float32),
        rng.integers(0, 2**31 - 1, 200_000, dtype=np.int64).astype(np.uint32).view(np.float32),
    ]
    v = np.concatenate(parts)
    v = v[np.isfinite(v)]
    ours = oracle.e4m3_encode(v)
    lib = np.clip(v, -448, 448).astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(ours, lib)


def test_brute_force_nearest_grid():
    grid_codes = np.arange(0x7F, dtype=np.uint8)
    grid = oracle.e4m3_decode(grid_codes)  # exact (table-driven, pinned above)
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.uniform(0, 460, 3000), rng.uniform(0, 2.0 ** -5, 3000)]).astype(np.float32)
    got = oracle.e4m3_encode(v)
    for x, c in zip(v.astype(np.float64), got):
        if x >= 448:
            assert c == 0x7E
            continue
        d = np.abs(grid - x)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert c == want, (x, c, want)


def test_negative_values_rounding_to_zero_keep_sign():
    v = np.array([-2.0 ** -11, -2.0 ** -10, -1e-30], dtype=np.float32)
    assert np.all(oracle.e4m3_encode(v) == 0x80)
