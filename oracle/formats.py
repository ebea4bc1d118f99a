"""Encoders and decoders of the read-copy storage formats, from the format definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The read copy is the low-precision copy of the checkpoint that non-flush steps read
instead of the FP32 checkpoint. Source: the blog post "ReplaySSM: Rethinking State
Storage for Faster Hybrid-Model Decoding", section "Benefit 3: Limit error accumulation
with separate precisions" (a flush casts the new high-precision checkpoint independently
into both formats; the copy never re-enters the recurrence). The pages fix neither the
rounding nor the scale; the readings taken here are:

* bf16: 1 sign, 8 exponent, 7 fraction bits (the top half of an IEEE binary32);
  round to nearest, ties to even.
* FP8 E4M3 as in the OCP 8-bit floating point specification (OFP8): 1 sign, 4 exponent
  (bias 7), 3 fraction bits; exponent field 0 holds subnormals m * 2**-9; S.1111.111 is
  NaN; no infinities; largest finite value 448. Round to nearest, ties to even, and
  saturate finite values beyond 448 to +-448.
* One FP32 scale per (sequence, head) slab: ``scale = absmax / 448`` (``1`` when the slab
  is all zero); codes ``q = e4m3(h / scale)``; the value read back is ``decode(q) * scale``.
  Both divisions are single IEEE binary32 divisions, so the code of each element is
  decided in FP32.
* NVFP4 (the post's sections "Benefit 3" and "State quantization" name it; the format is
  NVIDIA's published 4-bit block format): E2M1 elements (1 sign, 2 exponent bits with
  bias 1, 1 fraction bit; exponent field 0 holds 0 and 0.5; largest value 6; no inf or
  NaN), one E4M3 scale per block of 16 consecutive elements of a row, and one FP32 scale
  per tensor -- here per (sequence, head) slab, like the E4M3 copy. The scales follow the
  usual two-level recipe, each step one FP32 operation:
  ``s_g = absmax / (448 * 6)`` (``1`` for an all-zero slab); for each block
  ``s_b = e4m3(block_absmax / (6 * s_g))``; ``e = decode(s_b) * s_g``; codes
  ``q = e2m1(h / e)`` (round to nearest, ties to even, saturating at +-6), or 0 for the
  whole block when ``e`` is 0; the value read back is ``decode(q) * e``. Two codes share a
  byte, the even element in the low nibble.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_encode", "bf16_decode", "e4m3_decode", "e4m3_encode",
    "E4M3_MAX", "fp8_slab_quantize", "fp8_slab_dequantize",
    "E2M1_MAX", "NVFP4_BLOCK", "e2m1_decode", "e2m1_encode", "nvfp4_slab_quantize",
    "nvfp4_slab_dequantize", "nvfp4_pack", "nvfp4_unpack", "nvfp4_round_state",
]

E4M3_MAX = 448.0


def bf16_decode(bits) -> np.ndarray:
    """bf16 bit patterns -> FP32 values (exact: append 16 zero bits)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def bf16_encode(v) -> np.ndarray:
    """FP32 -> bf16 bit patterns, round to nearest, ties to even.

    For each finite ``v`` take the two bf16 neighbours that bracket it (``lo``: the
    FP32 bits with the low 16 bits cleared, i.e. truncation toward zero; ``hi``: the next
    bf16 away from zero), compare the two exact distances in FP64 and keep the nearer;
    on a tie keep the one whose last fraction bit is 0. A magnitude that rounds past the
    largest finite bf16 becomes infinity; NaN becomes the quiet NaN 0x7FC0 (with sign).
    """
    f = np.ascontiguousarray(v, dtype=np.float32)
    u = f.view(np.uint32)
    sign = (u >> np.uint32(16)) & np.uint32(0x8000)
    mag = u & np.uint32(0x7FFFFFFF)
    lo = mag >> np.uint32(16)                          # truncated magnitude, bf16 bits
    hi = lo + np.uint32(1)
    x = np.abs(f.astype(np.float64))
    lo_v = bf16_decode(np.minimum(lo, 0x7F7F).astype(np.uint16)).astype(np.float64)
    # Above the largest finite bf16 (0x7F7F) the next step of the binade would be 2**128;
    # RNE rounds to infinity from the midpoint up, so measure against 2**128 there.
    hi_v = np.where(hi >= 0x7F80, 2.0 ** 128,
                    bf16_decode(np.minimum(hi, 0x7F7F).astype(np.uint16)).astype(np.float64))
    with np.errstate(invalid="ignore"):
        d_lo = x - lo_v
        d_hi = hi_v - x
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((lo & np.uint32(1)) == 1))
    out = np.where(pick_hi, hi, lo)
    out = np.where(mag > np.uint32(0x7F800000), np.uint32(0x7FC0), out)      # NaN
    out = np.where(mag == np.uint32(0x7F800000), np.uint32(0x7F80), out)     # inf stays inf
    return (out | sign).astype(np.uint16)


def e4m3_decode(codes) -> np.ndarray:
    """OCP E4M3 codes -> FP64 values (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = m * 2.0 ** -9
    v = s * np.where(e == 0, sub, normal)
    return np.where((e == 15) & ((c & 0x7) == 7), np.nan, v)


_POS = e4m3_decode(np.arange(0x7F, dtype=np.uint8))    # codes 0x00..0x7E, ascending


def e4m3_encode(v) -> np.ndarray:
    """FP32 -> OCP E4M3 codes: round to nearest, ties to even, saturate to +-448.

    The nearest of the 127 finite non-negative values is found by search over the
    decoded table; on a tie the even code (fraction lsb 0) wins. The sign bit is kept,
    zero included. NaN maps to 0x7F (with sign).
    """
    f = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(f)
    i = np.clip(np.searchsorted(_POS, a, side="left"), 1, len(_POS) - 1)
    lo, hi = _POS[i - 1], _POS[i]
    with np.errstate(invalid="ignore"):
        d_lo, d_hi = a - lo, hi - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (((i - 1) & 1) == 1))
    code = np.where(pick_hi, i, i - 1)
    code = np.where(a >= E4M3_MAX, 0x7E, code)
    code = np.where(np.isnan(f), 0x7F, code)
    code = code | np.where(np.signbit(f), 0x80, 0)
    return code.astype(np.uint8)


def fp8_slab_quantize(h) -> tuple[np.ndarray, np.float32]:
    """Quantize one FP32 slab to (E4M3 codes, FP32 scale) with a per-slab absmax scale."""
    h = np.asarray(h, dtype=np.float32)
    absmax = np.float32(np.max(np.abs(h))) if h.size else np.float32(0)
    scale = np.float32(1.0) if absmax == 0 else np.float32(absmax / np.float32(E4M3_MAX))
    return e4m3_encode((h / scale).astype(np.float32)), scale


def fp8_slab_dequantize(codes, scale) -> np.ndarray:
    """Value read back from a slab's codes: decode(q) * scale, in FP32."""
    return (e4m3_decode(codes).astype(np.float32) * np.float32(scale)).astype(np.float32)


def bf16_round_state(h) -> np.ndarray:
    """A state rounded to bf16 element by element (FP64 -> FP32 -> bf16 RNE), widened back."""
    return bf16_decode(bf16_encode(np.asarray(h, dtype=np.float64).astype(np.float32))).astype(np.float64)


def e4m3_round_state(h) -> np.ndarray:
    """A state [..., P, N] rounded to E4M3 with one absmax scale per P x N slab, widened back."""
    h32 = np.asarray(h, dtype=np.float64).astype(np.float32)
    out = np.empty(h32.shape, dtype=np.float64)
    lead = h32.shape[:-2]
    for idx in np.ndindex(*lead):
        q, s = fp8_slab_quantize(h32[idx])
        out[idx] = fp8_slab_dequantize(q, s)
    return out


# ---------------------------------------------------------------------------------------
# IEEE binary16 (FP16): 1 sign, 5 exponent (bias 15), 10 fraction bits; exponent field 0
# holds subnormals m * 2**-24; largest finite value 65504.

def fp16_decode(bits) -> np.ndarray:
    """FP16 bit patterns -> FP64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    s = np.where(b & 0x8000, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    m = (b & 0x3FF).astype(np.float64)
    v = np.where(e == 0, m * 2.0 ** -24, (1.0 + m / 1024.0) * np.exp2(e.astype(np.float64) - 15.0))
    v = np.where(e == 31, np.where(m == 0, np.inf, np.nan), v)
    return s * v


_F16_POS = fp16_decode(np.arange(0x7C00, dtype=np.uint16))   # finite non-negative, ascending
FP16_MAX = 65504.0


def fp16_neighbours(v):
    """For FP32 values v: the FP16 code toward zero (lo) and the code next away from zero
    (hi), as bit patterns with v's sign, and their magnitudes. Past 65504 both are 65504."""
    f = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(f)
    i = np.searchsorted(_F16_POS, a, side="right") - 1          # largest code <= |v|
    i = np.clip(i, 0, len(_F16_POS) - 1)
    j = np.minimum(i + 1, len(_F16_POS) - 1)
    sign = np.where(np.signbit(f), 0x8000, 0)
    return ((i | sign).astype(np.uint16), (j | sign).astype(np.uint16), _F16_POS[i], _F16_POS[j])


def fp16_encode(v) -> np.ndarray:
    """FP32 -> FP16 codes, round to nearest, ties to even; finite values past the largest
    step round to infinity (IEEE)."""
    lo, hi, lv, hv = fp16_neighbours(v)
    a = np.abs(np.asarray(v, dtype=np.float32).astype(np.float64))
    top = (lo & 0x7FFF) == 0x7BFF
    hv = np.where(top, 65536.0, hv)                              # the next step past 65504
    d_lo, d_hi = a - lv, hv - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((lo & 1) == 1))
    out = np.where(pick_hi, np.where(top, (lo & 0x8000) | 0x7C00, hi), lo)
    return out.astype(np.uint16)


def fp16_sr_encode(v, u) -> np.ndarray:
    """FP32 -> FP16 codes by stochastic rounding: with lo and hi the FP16 neighbours of v
    (toward zero / away from zero), round to hi iff u < (|v| - |lo|) / (|hi| - |lo|), u in
    [0, 1). The ratio is exact in FP32 (the step is a power of two), so the decision is the
    same in any precision. Values past 65504 saturate to +-65504."""
    lo, hi, lv, hv = fp16_neighbours(v)
    a = np.abs(np.asarray(v, dtype=np.float32).astype(np.float64))
    with np.errstate(invalid="ignore", divide="ignore"):
        frac = np.where(hv > lv, (a - lv) / (hv - lv), 0.0)
    return np.where(np.asarray(u, dtype=np.float64) < frac, hi, lo).astype(np.uint16)


# The random draws of stochastic rounding, 16 bits each, four per output of the splitmix64
# sequence (Steele, Lea and Flood, OOPSLA 2014) started at SR_SEED: draw idx is 16-bit chunk
# idx mod 4 of output idx // 4, the most significant chunk first, and u = chunk / 2**16 in
# [0, 1). For the checkpoint of slab `slab` (of `num_slabs`) written by flush number `epoch`,
# element `elem` of P*N takes draw idx = (epoch * num_slabs + slab) * (P*N) + elem. Sixteen
# bits are exact for every FP16 normal: there the fraction of the spacing is a multiple of
# 2**-13, so P(u < frac) = frac.
SR_SEED = 0x2545F4914F6CDD1D
_SM_GAMMA, _SM_M1, _SM_M2 = 0x9E3779B97F4A7C15, 0xBF58476D1CE4E5B9, 0x94D049BB133111EB


def splitmix64(seed: int, idx) -> np.ndarray:
    """Output idx (0-based) of the splitmix64 sequence whose state starts at seed."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + (np.asarray(idx, dtype=np.uint64) + np.uint64(1)) * np.uint64(_SM_GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_SM_M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_SM_M2)
        return z ^ (z >> np.uint64(31))


def sr_uniform(idx) -> np.ndarray:
    """u in [0, 1) (multiples of 2**-16) for draw indices idx (uint64)."""
    idx = np.asarray(idx, dtype=np.uint64)
    z = splitmix64(SR_SEED, idx // np.uint64(4))
    shift = np.uint64(48) - np.uint64(16) * (idx % np.uint64(4))
    return ((z >> shift) & np.uint64(0xFFFF)).astype(np.float64) * 2.0 ** -16


def fp16_sr_round_state(h, epoch: int, slabs, num_slabs: int) -> np.ndarray:
    """A state [b, H, P, N] rounded to FP16 by stochastic rounding, widened back: slab
    (b, h) has index slabs[b] * H + h among num_slabs (so a subset of sequences can be
    followed), and its draws are those of flush `epoch`."""
    h32 = np.asarray(h, dtype=np.float64).astype(np.float32)
    bsz, H, P, N = h32.shape
    slab = (np.asarray(slabs, dtype=np.uint64).reshape(-1, 1) * np.uint64(H) +
            np.arange(H, dtype=np.uint64).reshape(1, -1)).reshape(bsz, H, 1, 1)
    elem = np.arange(P * N, dtype=np.uint64).reshape(1, 1, P, N)
    idx = (np.uint64(epoch) * np.uint64(num_slabs) + slab) * np.uint64(P * N) + elem
    return fp16_decode(fp16_sr_encode(h32, sr_uniform(idx)))


# ---------------------------------------------------------------------------------------
# NVFP4: E2M1 codes with a two-level scale (readings in the module docstring).
E2M1_MAX = 6.0
NVFP4_BLOCK = 16
_E2M1_POS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])   # codes 0..7 by definition


def e2m1_decode(codes) -> np.ndarray:
    """E2M1 codes (low 4 bits) -> FP64 values: sign bit 3, exponent bits 2..1 (bias 1),
    fraction bit 0; exponent 0 is subnormal (fraction * 0.5)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64) & 0xF
    e = (c >> 1) & 0x3
    m = (c & 0x1).astype(np.float64)
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e.astype(np.float64) - 1.0))
    return np.where(c & 0x8, -mag, mag)


def e2m1_encode(v) -> np.ndarray:
    """FP32 -> E2M1 codes: round to nearest, ties to even (fraction bit 0), saturate to
    +-6. The sign bit is kept, zero included."""
    f = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(f)
    i = np.clip(np.searchsorted(_E2M1_POS, a, side="left"), 1, len(_E2M1_POS) - 1)
    lo, hi = _E2M1_POS[i - 1], _E2M1_POS[i]
    d_lo, d_hi = a - lo, hi - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (((i - 1) & 1) == 1))
    code = np.where(pick_hi, i, i - 1)
    code = np.where(a >= E2M1_MAX, 7, code)
    return (code | np.where(np.signbit(f), 0x8, 0)).astype(np.uint8)


def nvfp4_slab_quantize(h):
    """One FP32 slab [P, N] -> (E2M1 codes [P, N], E4M3 block-scale codes [P, N/16],
    FP32 slab scale). Every step is the single FP32 operation the recipe states."""
    h = np.asarray(h, dtype=np.float32)
    P, N = h.shape
    absmax = np.float32(np.max(np.abs(h))) if h.size else np.float32(0)
    s_g = np.float32(1.0) if absmax == 0 else np.float32(absmax / np.float32(E4M3_MAX * E2M1_MAX))
    blocks = h.reshape(P, N // NVFP4_BLOCK, NVFP4_BLOCK)
    bmax = np.max(np.abs(blocks), axis=2).astype(np.float32)
    s_b = e4m3_encode((bmax / (np.float32(E2M1_MAX) * s_g)).astype(np.float32))
    e = (e4m3_decode(s_b).astype(np.float32) * s_g).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (blocks / e[:, :, None]).astype(np.float32)
    q = np.where(e[:, :, None] > 0, e2m1_encode(r), 0).astype(np.uint8)
    return q.reshape(P, N), s_b, s_g


def nvfp4_slab_dequantize(q, s_b, s_g) -> np.ndarray:
    """Value read back: decode(q) * (decode(s_b) * s_g), with the block scale product in
    FP32 as in the recipe (the element product is exact in FP64)."""
    q = np.asarray(q, dtype=np.uint8)
    P, N = q.shape
    e = (e4m3_decode(s_b).astype(np.float32) * np.float32(s_g)).astype(np.float64)
    return (e2m1_decode(q).reshape(P, N // NVFP4_BLOCK, NVFP4_BLOCK) * e[:, :, None]).reshape(P, N)


def nvfp4_pack(q) -> np.ndarray:
    """Codes [..., N] -> bytes [..., N/2]: element 2j in the low nibble, 2j+1 in the high."""
    q = np.asarray(q, dtype=np.uint8)
    return (q[..., 0::2] & 0xF) | ((q[..., 1::2] & 0xF) << 4)


def nvfp4_unpack(b) -> np.ndarray:
    """Bytes [..., N/2] -> codes [..., N]."""
    b = np.asarray(b, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = b >> 4
    return out


def nvfp4_round_state(h) -> np.ndarray:
    """A state [..., P, N] quantized slab by slab to NVFP4 and read back (FP64)."""
    h32 = np.asarray(h, dtype=np.float64).astype(np.float32)
    out = np.empty(h32.shape, dtype=np.float64)
    for idx in np.ndindex(*h32.shape[:-2]):
        out[idx] = nvfp4_slab_dequantize(*nvfp4_slab_quantize(h32[idx]))
    return out
