"""Pins of the oracle's E4M3 and E2M1 codecs against the format definitions.

The E4M3 table is pinned by printed landmark codes, its size, NaN codes and
monotonicity; the encoder by round trips, every midpoint, and an exhaustive
comparison over all 2^32 fp32 patterns with a nearest-value search over the
decoded table (which uses no encoder arithmetic).
"""
import math
import struct

import numpy as np
import pytest

from conftest import read_golden


def f32_bits(x):
    return struct.unpack("<I", struct.pack("<f", x))[0]


def f32_from_bits(b):
    return struct.unpack("<f", struct.pack("<I", b))[0]


def test_e4m3_landmarks(orc):
    for code, val in read_golden("e4m3_landmarks.txt"):
        got = orc.lib().orc_e4m3_decode(int(code, 16))
        if val == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(val), (code, got, val)
            if val == "-0.0":
                assert math.copysign(1.0, got) < 0


def test_e4m3_table_shape(orc):
    vals = [orc.lib().orc_e4m3_decode(c) for c in range(256)]
    nans = [c for c, v in enumerate(vals) if math.isnan(v)]
    assert nans == [0x7F, 0xFF]
    finite = [v for v in vals if not math.isnan(v)]
    assert len(finite) == 254
    pos = vals[0:0x7F]
    assert all(b > a for a, b in zip(pos, pos[1:])), "positive codes strictly increasing"
    assert max(finite) == 448.0 and min(finite) == -448.0
    # the negative half mirrors the positive half
    for c in range(0x7F):
        assert vals[c | 0x80] == -vals[c]


def test_e4m3_roundtrip(orc):
    L = orc.lib()
    for c in range(256):
        v = L.orc_e4m3_decode(c)
        if math.isnan(v):
            continue
        assert L.orc_e4m3_encode(v) == c, hex(c)


def test_e4m3_midpoints_ties_to_even(orc):
    L = orc.lib()
    pos = [L.orc_e4m3_decode(c) for c in range(0x7F)]
    for c in range(0x7E):
        lo, hi = pos[c], pos[c + 1]
        mid = (lo + hi) / 2.0           # exact in fp32 for E4M3 neighbours
        assert np.float32(mid) == mid
        even = c if c % 2 == 0 else c + 1
        assert L.orc_e4m3_encode(mid) == even, hex(c)
        assert L.orc_e4m3_encode(-mid) == even | 0x80
        below = float(np.nextafter(np.float32(mid), np.float32(0)))
        above = float(np.nextafter(np.float32(mid), np.float32(1e9)))
        assert L.orc_e4m3_encode(below) == c
        assert L.orc_e4m3_encode(above) == c + 1


def test_e4m3_saturation_and_zero(orc):
    L = orc.lib()
    for x in [448.0, 449.0, 463.9, 464.0, 465.0, 1e6, 3.4e38, float("inf")]:
        assert L.orc_e4m3_encode(x) == 0x7E
        assert L.orc_e4m3_encode(-x) == 0xFE
    assert L.orc_e4m3_encode(0.0) == 0x00
    assert L.orc_e4m3_encode(-0.0) == 0x80
    assert L.orc_e4m3_encode(-1e-30) == 0x80
    assert L.orc_e4m3_encode(2.0 ** -10) == 0x00   # tie between 0 and 2^-9 -> even (0)
    assert L.orc_e4m3_encode(f32_from_bits(f32_bits(2.0 ** -10) + 1)) == 0x01


def test_e2m1_grid(orc):
    L = orc.lib()
    for code, val in read_golden("e2m1_grid.txt"):
        got = L.orc_e2m1_decode(int(code, 16))
        assert got == float(val)
        if val.startswith("-"):
            assert math.copysign(1.0, got) < 0
    for c in range(16):
        assert L.orc_e2m1_encode(L.orc_e2m1_decode(c)) == c


def test_e2m1_ties(orc):
    L = orc.lib()
    # midpoints of the grid go to the neighbour with the even code
    table = {0.25: 0x0, 0.75: 0x2, 1.25: 0x2, 1.75: 0x4, 2.5: 0x4, 3.5: 0x6, 5.0: 0x6}
    for x, c in table.items():
        assert L.orc_e2m1_encode(x) == c, x
        assert L.orc_e2m1_encode(-x) == c | 0x8, x
        below = float(np.nextafter(np.float32(x), np.float32(0)))
        above = float(np.nextafter(np.float32(x), np.float32(100)))
        lo = {0.25: 0x0, 0.75: 0x1, 1.25: 0x2, 1.75: 0x3, 2.5: 0x4, 3.5: 0x5, 5.0: 0x6}[x]
        assert L.orc_e2m1_encode(below) == lo
        assert L.orc_e2m1_encode(above) == lo + 1
    for x in [6.0, 6.5, 7.0, 1e30, float("inf")]:
        assert L.orc_e2m1_encode(x) == 0x7
        assert L.orc_e2m1_encode(-x) == 0xF
    assert L.orc_e2m1_encode(-0.0) == 0x8
    assert L.orc_e2m1_encode(-0.2) == 0x8


def test_vector_encoders_match_scalar(orc):
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(4096) * rng.choice([1e-3, 1, 100, 1e4], 4096)).astype(np.float32)
    e = orc.e4m3_encode(x)
    f = orc.e2m1_encode(x)
    L = orc.lib()
    for i in range(0, 4096, 97):
        assert e[i] == L.orc_e4m3_encode(float(x[i]))
        assert f[i] == L.orc_e2m1_encode(float(x[i]))


@pytest.mark.parametrize("kind", [0, 1], ids=["e4m3", "e2m1"])
def test_encoder_exhaustive_vs_table_search(orc, kind):
    """All 2^32 fp32 patterns (NaNs skipped): encoder == nearest table value."""
    bad, first = orc.bruteforce_encode_check(kind, 0, 1 << 32)
    assert bad == 0, f"{bad} mismatches, first pattern {first:#010x}"
