"""Seeded synthetic inputs for a Mamba-2 decode layer.

This module is shared by the CUDA library's tests and benchmark and by the FP64
oracle. It holds no arithmetic of the decode method itself: only a counter-based
random generator, the value distributions of the workloads, and rounding of the
drawn values to the storage dtype (FP32 or bf16).

Generator. Value ``i`` of stream ``s`` under seed ``k`` is the ``i``-th output of a
splitmix64 sequence (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) whose state starts at ``mix64(k * gamma + s)``. Every value
is therefore a pure function of ``(k, s, i)``: any subset of sequences, heads or
tokens can be drawn without drawing the rest. Uniforms take the top 53 bits,
``(z >> 11 + 0.5) * 2**-53`` in (0, 1); normals use the Box-Muller cosine branch on
uniforms ``2i`` and ``2i + 1``.

Index layout. The index of a per-token value depends on the sequence ``b`` and the
token ``t`` but not on the batch size, so sequence ``b`` sees the same inputs in a
batch of 1 and in a batch of 512:

* ``x[b, t, h, p]``   -> ``((b * 2**20 + t) * H + h) * P + p``
* ``B/C[b, t, g, n]`` -> ``((b * 2**20 + t) * G + g) * N + n``
* ``dt[b, t, h]``     -> ``(b * 2**20 + t) * H + h``

Distributions (the Mamba-2 decode workloads; values drawn in FP64, rounded RNE to
FP32, then RNE to bf16 where the inputs are bf16):

* ``x ~ N(0, 1)``;  ``B, C ~ N(0, 1) / sqrt(N)``;
* ``dt = softplus(z - 2) = log1p(exp(z - 2))``, ``z ~ N(0, 1)``;
* ``A_h = -exp(U(0, ln 16))`` (so ``A_h`` lies in ``[-16, -1]``);  ``D_h ~ N(0, 1)``;
* an imported state ``h0 ~ 0.1 * N(0, 1)``;
* a speculative accept length ``a ~ U{0..T}``.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

__all__ = [
    "STREAM", "LayerShape", "uniform", "normal", "round_f32", "round_bf16_bits",
    "bf16_bits_to_f64", "head_params", "token_inputs", "draft_inputs",
    "initial_state", "accept_lengths",
]

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_TOKEN_STRIDE = 1 << 20          # tokens per sequence addressable in the index layout

STREAM = {
    "x": 1, "B": 2, "C": 3, "dt": 4, "A": 5, "D": 6, "accept": 7, "h0": 8,
    "xd": 11, "Bd": 12, "Cd": 13, "dtd": 14,    # speculative draft tokens
}


def _mix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function (wrapping uint64 arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _raw(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        base = _mix64(np.array([seed], dtype=np.uint64) * _GAMMA + np.uint64(stream))[0]
        state = base + (np.asarray(idx, dtype=np.uint64) + np.uint64(1)) * _GAMMA
        return _mix64(state)


def uniform(seed: int, stream: int, idx) -> np.ndarray:
    """U(0, 1) doubles, open at both ends."""
    z = _raw(seed, stream, idx)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(seed: int, stream: int, idx) -> np.ndarray:
    """N(0, 1) doubles (Box-Muller, cosine branch)."""
    idx = np.asarray(idx, dtype=np.uint64)
    u1 = uniform(seed, stream, idx * np.uint64(2))
    u2 = uniform(seed, stream, idx * np.uint64(2) + np.uint64(1))
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def round_f32(v: np.ndarray) -> np.ndarray:
    """FP64 -> FP32, round to nearest even (numpy's cast)."""
    return np.asarray(v, dtype=np.float64).astype(np.float32)


def round_bf16_bits(v: np.ndarray) -> np.ndarray:
    """FP64 -> FP32 (RNE) -> bf16 (RNE); returns the bf16 bit patterns as uint16.

    The inputs are finite, so the carry trick on the FP32 bits is exact RNE here.
    """
    bits = round_f32(v).view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    return ((bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@dataclass(frozen=True)
class LayerShape:
    """Shape of one Mamba-2 layer's decode inputs; ``dtype`` is 'f32' or 'bf16'."""
    batch: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    dtype: str = "f32"

    def __post_init__(self):
        if self.nheads % self.ngroups:
            raise ValueError("nheads must be a multiple of ngroups")
        if self.dtype not in ("f32", "bf16"):
            raise ValueError("dtype must be 'f32' or 'bf16'")


class Drawn:
    """One tensor of inputs: ``store`` is what a device consumes (float32, or uint16
    bf16 bits), ``f64`` is the very same values widened to FP64."""
    __slots__ = ("store", "f64")

    def __init__(self, v64: np.ndarray, dtype: str):
        if dtype == "f32":
            self.store = round_f32(v64)
            self.f64 = self.store.astype(np.float64)
        else:
            self.store = round_bf16_bits(v64)
            self.f64 = bf16_bits_to_f64(self.store)


def head_params(nheads: int, seed: int):
    """Per-head decay rate A (< 0) and skip weight D, both FP32; returns float32 arrays."""
    h = np.arange(nheads, dtype=np.uint64)
    A = -np.exp(uniform(seed, STREAM["A"], h) * np.log(16.0))
    D = normal(seed, STREAM["D"], h)
    return round_f32(A), round_f32(D)


def _token_index(seqs, toks, inner):
    seqs = np.asarray(seqs, dtype=np.uint64).reshape(-1, 1, 1)
    toks = np.asarray(toks, dtype=np.uint64).reshape(1, -1, 1)
    inner = np.uint64(inner)
    row = (seqs * np.uint64(_TOKEN_STRIDE) + toks) * inner
    return row + np.arange(inner, dtype=np.uint64).reshape(1, 1, -1)


def _draw_tokens(shape: LayerShape, seed: int, seqs, toks, names):
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    nb, nt = len(seqs), len(toks)
    sx, sb, sc, sd = (STREAM[n] for n in names)
    x = normal(seed, sx, _token_index(seqs, toks, H * P)).reshape(nb, nt, H, P)
    B = normal(seed, sb, _token_index(seqs, toks, G * N)).reshape(nb, nt, G, N) / np.sqrt(N)
    C = normal(seed, sc, _token_index(seqs, toks, G * N)).reshape(nb, nt, G, N) / np.sqrt(N)
    z = normal(seed, sd, _token_index(seqs, toks, H)).reshape(nb, nt, H)
    dt = np.log1p(np.exp(z - 2.0))
    return {k: Drawn(v, shape.dtype) for k, v in (("x", x), ("B", B), ("C", C), ("dt", dt))}


def token_inputs(shape: LayerShape, seed: int, toks, seqs=None):
    """Decode-token inputs for tokens ``toks`` of sequences ``seqs`` (default: all).

    Returns a dict of :class:`Drawn` with arrays shaped ``x[b, t, H, P]``,
    ``B/C[b, t, G, N]``, ``dt[b, t, H]``.
    """
    seqs = np.arange(shape.batch) if seqs is None else np.asarray(seqs)
    return _draw_tokens(shape, seed, seqs, np.atleast_1d(toks), ("x", "B", "C", "dt"))


def draft_inputs(shape: LayerShape, seed: int, call: int, T: int, seqs=None):
    """Inputs of the ``T`` draft tokens of speculative call ``call`` (own streams)."""
    seqs = np.arange(shape.batch) if seqs is None else np.asarray(seqs)
    toks = call * T + np.arange(T)
    return _draw_tokens(shape, seed, seqs, toks, ("xd", "Bd", "Cd", "dtd"))


def initial_state(shape: LayerShape, seed: int, seqs=None) -> np.ndarray:
    """An imported FP32 state ``h0[b, H, P, N] ~ 0.1 * N(0, 1)``."""
    seqs = np.arange(shape.batch) if seqs is None else np.asarray(seqs)
    H, P, N = shape.nheads, shape.headdim, shape.dstate
    inner = H * P * N
    idx = np.asarray(seqs, dtype=np.uint64).reshape(-1, 1) * np.uint64(inner) + \
        np.arange(inner, dtype=np.uint64).reshape(1, -1)
    return round_f32(0.1 * normal(seed, STREAM["h0"], idx)).reshape(len(seqs), H, P, N)


def accept_lengths(batch: int, T: int, seed: int, call: int) -> np.ndarray:
    """Accepted draft counts ``a_b ~ U{0..T}`` for speculative call ``call`` (int32)."""
    idx = np.arange(batch, dtype=np.uint64) * np.uint64(_TOKEN_STRIDE) + np.uint64(call)
    a = np.floor(uniform(seed, STREAM["accept"], idx) * (T + 1)).astype(np.int32)
    return np.minimum(a, T)
