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


def test_state_rounding_helpers():
    rng = np.random.default_rng(5)
    h = rng.standard_normal((2, 3, 4, 8))
    hb = F.bf16_round_state(h)
    assert np.array_equal(hb, F.bf16_decode(F.bf16_encode(h.astype(np.float32))))
    he = F.e4m3_round_state(h)
    for b in range(2):
        for k in range(3):
            q, s = F.fp8_slab_quantize(h[b, k].astype(np.float32))
            assert np.array_equal(he[b, k], F.fp8_slab_dequantize(q, s))


def test_fp16_code_points_roundtrip_and_ties():
    assert F.fp16_decode(np.uint16(0x3C00)) == 1.0 and F.fp16_decode(np.uint16(0x7BFF)) == 65504.0
    assert F.fp16_decode(np.uint16(0x0001)) == 2.0 ** -24 and F.fp16_decode(np.uint16(0x0400)) == 2.0 ** -14
    assert np.isinf(F.fp16_decode(np.uint16(0x7C00))) and np.isnan(F.fp16_decode(np.uint16(0x7E00)))
    p = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = p[((p.astype(np.uint32) >> 10) & 0x1F) != 0x1F]
    assert np.array_equal(F.fp16_encode(F.fp16_decode(finite).astype(np.float32)), finite)
    pos = np.arange(0x7C00, dtype=np.uint16)
    v = F.fp16_decode(pos)
    mid = ((v[:-1] + v[1:]) / 2).astype(np.float32)        # exact in FP32
    even = np.where(pos[:-1] & 1, pos[:-1] + 1, pos[:-1]).astype(np.uint16)
    assert np.array_equal(F.fp16_encode(mid), even)
    assert F.fp16_encode(np.float32(65520.0)) == 0x7C00    # midpoint past 65504 -> inf
    assert F.fp16_encode(np.float32(65519.0)) == 0x7BFF


def test_fp16_stochastic_rounding_definition():
    lo_hi = F.fp16_decode(np.array([0x3C00, 0x3C01], dtype=np.uint16))   # 1 and 1 + 2**-10
    v = np.float32(1.0 + 0.25 * 2.0 ** -10)                               # a quarter of the way
    assert F.fp16_sr_encode(v, 0.0) == 0x3C01 and F.fp16_sr_encode(v, 0.2499) == 0x3C01
    assert F.fp16_sr_encode(v, 0.25) == 0x3C00 and F.fp16_sr_encode(v, 0.9) == 0x3C00
    assert F.fp16_sr_encode(-v, 0.1) == 0xBC01                            # sign kept
    exact = F.fp16_decode(np.arange(0, 0x7C00, 97, dtype=np.uint16)).astype(np.float32)
    assert np.array_equal(F.fp16_decode(F.fp16_sr_encode(exact, 0.0)), exact)   # no bias on grid points
    assert F.fp16_sr_encode(np.float32(1e6), 0.0) == 0x7BFF                     # saturates
    # unbiased: the mean over uniform draws is the value itself
    u = F.sr_uniform(np.arange(200000, dtype=np.uint64))
    assert abs(u.mean() - 0.5) < 0.003 and u.min() >= 0 and u.max() < 1
    vals = F.fp16_decode(F.fp16_sr_encode(np.full(200000, 1.0 + 0.3 * 2.0 ** -10, np.float32), u))
    assert abs(vals.mean() - (1.0 + 0.3 * 2.0 ** -10)) < 2e-6
    assert set(np.unique(vals)) <= set(lo_hi)


def test_splitmix64_reference_values():
    """The first outputs of the published generator started at 0, and the 16-bit draws cut
    from them, most significant chunk first."""
    z = F.splitmix64(0, np.arange(3))
    assert [int(v) for v in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    w = int(F.splitmix64(F.SR_SEED, [1])[0])                 # the output that draws 4..7 come from
    got = F.sr_uniform(np.arange(4, 8, dtype=np.uint64)) * 2.0 ** 16
    assert got.tolist() == [(w >> 48) & 0xFFFF, (w >> 32) & 0xFFFF, (w >> 16) & 0xFFFF, w & 0xFFFF]


# ------------------------------------------------------------------ NVFP4
# The E2M1 value set as the format's published tables list it (codes 0..7; 8..15 are the
# negatives): 0, 0.5, 1, 1.5, 2, 3, 4, 6.
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_code_points_and_roundtrip():
    codes = np.arange(16, dtype=np.uint8)
    want = np.array(E2M1_TABLE + [-v for v in E2M1_TABLE])
    got = F.e2m1_decode(codes)
    assert np.array_equal(got, want)
    assert np.all(np.signbit(got[8:]))                       # code 8 is -0
    assert np.array_equal(F.e2m1_encode(got.astype(np.float32)), codes)


def test_e2m1_ties_to_even_nearest_and_saturation():
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    want = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]               # the neighbour with fraction bit 0
    assert F.e2m1_decode(F.e2m1_encode(mids)).tolist() == want
    assert F.e2m1_decode(F.e2m1_encode(-mids)).tolist() == [-w for w in want]
    near = np.array([0.26, 0.74, 1.3, 2.49, 2.51, 3.4, 4.9, 5.1, 6.0, 7.0, 1e30], dtype=np.float32)
    assert F.e2m1_decode(F.e2m1_encode(near)).tolist() == [0.5, 0.5, 1.5, 2.0, 3.0, 3.0, 4.0, 6.0, 6.0, 6.0, 6.0]
    assert F.e2m1_encode(np.float32(-1e-9)) == 0x8              # sign kept on zero


def test_nvfp4_pack_nibble_order():
    q = np.array([[2, 7, 0, 15]], dtype=np.uint8)               # 1.0, 6.0, 0, -6.0
    b = F.nvfp4_pack(q)
    assert b.tolist() == [[0x72, 0xF0]]
    assert np.array_equal(F.nvfp4_unpack(b), q)


def test_nvfp4_exactly_representable_slab():
    """A slab built from E2M1 values times block scales that E4M3 holds exactly, with the
    slab's absmax 448 * 6 * s_g: every code comes back exactly and every value to FP32
    rounding."""
    rng = np.random.default_rng(3)
    P, N = 8, 64
    s_g = np.float32(1.0 / 4096)                              # a power of two: products exact
    bs_vals = F.e4m3_decode(np.arange(0x38, 0x7F, dtype=np.uint8))   # 1 .. 448
    s_b = rng.choice(bs_vals, size=(P, N // 16))
    s_b[0, 0] = 448.0
    k = rng.integers(0, 16, size=(P, N)).astype(np.uint8)
    k[0, 0] = 7                                              # the slab's absmax: 6 * 448 * s_g
    for blk in np.ndindex(P, N // 16):                       # each block reaches +-6 once
        k[blk[0], blk[1] * 16] = 7
    h = (F.e2m1_decode(k).reshape(P, N // 16, 16) * (s_b * s_g)[:, :, None]).reshape(P, N)
    q, sb, sg = F.nvfp4_slab_quantize(h.astype(np.float32))
    assert sg == s_g
    assert np.array_equal(F.e4m3_decode(sb), s_b)
    assert np.array_equal(F.e2m1_decode(q), F.e2m1_decode(k))
    assert np.array_equal(F.nvfp4_slab_dequantize(q, sb, sg), h)


def test_nvfp4_zero_slab_and_zero_block():
    q, sb, sg = F.nvfp4_slab_quantize(np.zeros((4, 32), np.float32))
    assert sg == 1.0 and not q.any() and not sb.any()
    h = np.zeros((4, 32), np.float32)
    h[0, 0] = 1.0
    h[1, 17] = 1e-9                                          # far below the block-scale range
    q, sb, sg = F.nvfp4_slab_quantize(h)
    assert sb[1, 1] == 0 and not q[1, 16:].any()              # a zero scale zeroes the block
    assert F.e2m1_decode(q[0, 0]) == 6.0 and F.e4m3_decode(sb[0, 0]) == 448.0


def test_nvfp4_error_bound_on_random_slabs():
    """Each value read back is within one E2M1 step of the block's scale unit e (the
    largest half step, between 4 and 6, is 1 * e), and a block's absmax within 1/8 of
    itself (a normal E4M3 scale is within 2**-4 of exact, then E2M1 saturates at 6; these
    Gaussian slabs keep every block scale in the normal range)."""
    rng = np.random.default_rng(5)
    for trial in range(20):
        h = (rng.standard_normal((16, 128)) * 10.0 ** rng.uniform(-6, 3)).astype(np.float32)
        q, sb, sg = F.nvfp4_slab_quantize(h)
        e = F.e4m3_decode(sb) * float(sg)
        back = F.nvfp4_slab_dequantize(q, sb, sg)
        err = np.abs(back - h).reshape(16, 8, 16)
        assert np.all(err <= e[:, :, None] * (1.0 + 1e-6)), trial
        bmax = np.abs(h).reshape(16, 8, 16).max(axis=2)
        bback = np.abs(back).reshape(16, 8, 16).max(axis=2)
        assert np.all(np.abs(bback - bmax) <= bmax / 8 + 1e-30), trial


# ------------------------------------------------------------------ state rounding of the shared checkpoints
def test_fp16_sr_state_draw_index_hand_worked():
    """The draw of element e of slab s written by flush `epoch` is output
    (epoch * num_slabs + s) * P*N + e of the generator, with s numbered over the whole batch
    (s = b * H + h for the sequence's place b in the batch, not its place in the subset
    followed). Here the oracle follows sequences 4 and 1 of a 5-sequence batch (H = 3,
    P = 2, N = 4, so num_slabs = 15 and P*N = 8) at epoch 2. Six elements sit a hair above
    or below their own draw between the FP16 neighbours 1 and 1 + 2**-10 (times a power of
    two), so each rounds the way that draw alone decides; the rest are FP16 values, which
    stochastic rounding keeps whatever the draw."""
    H, P, N, epoch, num_slabs = 3, 2, 4, 2, 15
    # (place in the state, head, row, column) -> draw index, worked by hand:
    #   slab = seq * 3 + head, elem = row * 4 + column, idx = (2 * 15 + slab) * 8 + elem
    hand = {
        (0, 2, 1, 3): 359,   # seq 4: slab 14, elem 7 -> (30 + 14) * 8 + 7
        (1, 0, 0, 0): 264,   # seq 1: slab 3,  elem 0 -> (30 + 3) * 8 + 0
        (0, 0, 0, 1): 337,   # seq 4: slab 12, elem 1 -> (30 + 12) * 8 + 1
        (1, 2, 1, 2): 286,   # seq 1: slab 5,  elem 6 -> (30 + 5) * 8 + 6
        (0, 1, 0, 2): 346,   # seq 4: slab 13, elem 2 -> (30 + 13) * 8 + 2
        (1, 1, 1, 0): 276,   # seq 1: slab 4,  elem 4 -> (30 + 4) * 8 + 4
    }
    rng = np.random.default_rng(11)
    grid = F.fp16_decode(rng.integers(0x2000, 0x5000, size=(2, H, P, N)).astype(np.uint16))
    grid = np.where(rng.random(grid.shape) < 0.5, -grid, grid)
    h = grid.copy()
    want = grid.copy()
    for j, (pos, idx) in enumerate(sorted(hand.items())):
        u = F.sr_uniform(np.array([idx], dtype=np.uint64))[0]
        k = int(u * 2 ** 13)                       # the draw's first 13 bits: k / 2**13 <= u
        up = j % 2 == 0
        frac = (k + 1) / 2 ** 13 if up else k / 2 ** 13   # above the draw: rounds away from zero
        scale = 2.0 ** (j - 3) * (-1 if j == 3 else 1)
        h[pos] = scale * (1.0 + frac * 2.0 ** -10)         # exact in FP32 (13 fraction bits)
        want[pos] = scale * ((1.0 + 2.0 ** -10) if up else 1.0)
    got = F.fp16_sr_round_state(h, epoch, [4, 1], num_slabs)
    assert np.array_equal(got, want)


def test_nvfp4_state_rounding_is_per_slab():
    """A state of several slabs, each built (as in the exactly-representable test) from
    E2M1 values times E4M3-exact block scales under its own power-of-two slab scale, comes
    back exactly: each slab takes its own absmax scale and its blocks run along a row. One
    slab is zero and stays zero."""
    rng = np.random.default_rng(4)
    P, N = 16, 64
    bs_vals = F.e4m3_decode(np.arange(0x38, 0x7F, dtype=np.uint8))   # 1 .. 448
    h = np.zeros((2, 3, P, N))
    for b in range(2):
        for k in range(3):
            if (b, k) == (1, 2):
                continue                                          # the zero slab
            s_g = 2.0 ** -(6 + 3 * (3 * b + k))                   # a different scale per slab
            s_b = rng.choice(bs_vals, size=(P, N // 16))
            s_b[rng.integers(P), rng.integers(2)] = 448.0           # in the first 32 columns
            q = rng.integers(0, 16, size=(P, N)).astype(np.uint8)
            q[:, ::16] = np.where(rng.random((P, N // 16)) < 0.5, 7, 15)   # each block reaches +-6
            h[b, k] = (F.e2m1_decode(q).reshape(P, N // 16, 16) * (s_b * s_g)[:, :, None]).reshape(P, N)
    assert np.array_equal(F.nvfp4_round_state(h), h)
    assert np.array_equal(F.nvfp4_round_state(h[:, :, :, :32]), h[:, :, :, :32])   # a narrower slab
