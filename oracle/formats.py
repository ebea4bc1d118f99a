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
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_encode", "bf16_decode", "e4m3_decode", "e4m3_encode",
    "E4M3_MAX", "fp8_slab_quantize", "fp8_slab_dequantize",
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
