"""The read-copy format encoders against the format definitions (CPU, exhaustive)."""
import json
import pathlib

import numpy as np

from oracle import formats as F

GOLDEN = pathlib.Path(__file__).parent / "golden"


def _finite_bf16_patterns():
    p = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    exp = (p.astype(np.uint32) >> 7) & 0xFF
    return p[exp != 0xFF]


def test_bf16_roundtrip_all_finite():
    p = _finite_bf16_patterns()
    assert np.array_equal(F.bf16_encode(F.bf16_decode(p)), p)


def test_bf16_midpoints_tie_to_even_and_neighbours_round_to_nearest():
    p = _finite_bf16_patterns()
    pos = np.sort(p[(p < 0x7F80)])                      # 0 .. largest finite, ascending
    lo = pos[:-1].astype(np.uint32)
    lo_v = F.bf16_decode(pos[:-1]).astype(np.float64)
    hi_v = F.bf16_decode(pos[1:]).astype(np.float64)
    mid = ((lo_v + hi_v) / 2).astype(np.float32)       # exact: 8 more bits fit in FP32
    assert np.all(mid.astype(np.float64) == (lo_v + hi_v) / 2)
    even = np.where(lo & 1, lo + 1, lo).astype(np.uint16)
    assert np.array_equal(F.bf16_encode(mid), even)
    assert np.array_equal(F.bf16_encode(-mid), even | np.uint16(0x8000))
    below = np.nextafter(mid, np.float32(0))
    above = np.nextafter(mid, np.float32(np.inf))
    assert np.array_equal(F.bf16_encode(below), pos[:-1])
    assert np.array_equal(F.bf16_encode(above), pos[1:])


def test_bf16_specials():
    f = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 3.4028234663852886e38, -np.inf, np.nan, 0.0, -0.0],
                 dtype=np.float32)
    got = F.bf16_encode(f)
    assert got[0] == 0x3F80          # tie -> even (1.0)
    assert got[1] == 0x3F82          # tie between 0x3F81 and 0x3F82 -> even
    assert got[2] == 0x7F80          # FP32 max is past the bf16 overflow midpoint -> inf
    assert got[3] == 0xFF80
    assert got[4] == 0x7FC0
    assert got[5] == 0x0000 and got[6] == 0x8000
    top_mid = np.float32(2.0 ** 128 - 2.0 ** 119)      # midpoint of 0x7F7F and 2**128
    assert F.bf16_encode(top_mid) == 0x7F80
    assert F.bf16_encode(np.nextafter(top_mid, np.float32(0))) == 0x7F7F


def test_e4m3_code_points_from_ocp_spec():
    doc = json.loads((GOLDEN / "e4m3_ocp_values.json").read_text())
    for code, val in doc["codes"].items():
        v = F.e4m3_decode(np.uint8(int(code, 16)))
        assert v == val, (code, v, val)
    for code in doc["nan_codes"]:
        assert np.isnan(F.e4m3_decode(np.uint8(int(code, 16))))
    vals = F.e4m3_decode(np.arange(0x80, dtype=np.uint8))
    finite = vals[~np.isnan(vals)]
    assert len(finite) == doc["finite_nonnegative_count"]
    assert np.all(np.diff(finite) > 0)
    assert np.signbit(F.e4m3_decode(np.uint8(0x80)))


def test_e4m3_roundtrip_ties_and_saturation():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    v = F.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(F.e4m3_encode(v), codes)
    pos = F.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mid = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.all(mid.astype(np.float64) == (pos[:-1] + pos[1:]) / 2)
    i = np.arange(0x7E)
    even = np.where(i & 1, i + 1, i)
    assert np.array_equal(F.e4m3_encode(mid), even.astype(np.uint8))
    assert np.array_equal(F.e4m3_encode(np.nextafter(mid, np.float32(0))), i.astype(np.uint8))
    assert np.array_equal(F.e4m3_encode(np.nextafter(mid, np.float32(1e9))), (i + 1).astype(np.uint8))
    sat = np.array([448.0, 449.0, 464.0, 500.0, 1e30, np.inf], dtype=np.float32)
    assert np.all(F.e4m3_encode(sat) == 0x7E)
    assert np.all(F.e4m3_encode(-sat) == 0xFE)
    assert F.e4m3_encode(np.float32(np.nan)) & 0x7F == 0x7F
    assert F.e4m3_encode(np.float32(2 ** -11)) == 0x00       # below half the smallest subnormal
    assert F.e4m3_encode(np.float32(-2 ** -11)) == 0x80


def test_fp8_slab_scale_and_codes():
    rng = np.random.default_rng(0)
    h = (rng.standard_normal((64, 128)) * 0.3).astype(np.float32)
    q, s = F.fp8_slab_quantize(h)
    amax = np.float32(np.abs(h).max())
    assert s == np.float32(amax / np.float32(448.0))
    assert np.max(F.e4m3_decode(q & 0x7F)) == 448.0        # the absmax element lands on 448
    back = F.fp8_slab_dequantize(q, s)
    # E4M3 keeps 3 fraction bits: normal values are within 2**-4 relative
    big = np.abs(h) >= s * 2.0 ** -6
    assert np.all(np.abs(back[big] - h[big]) <= np.abs(h[big]) * 2.0 ** -4)
    z, s0 = F.fp8_slab_quantize(np.zeros((4, 4), np.float32))
    assert s0 == 1.0 and not np.any(z & 0x7F)
