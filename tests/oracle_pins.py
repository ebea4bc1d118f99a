"""Pins that tie the FP64 oracle to facts outside itself.

Each ``pin_*`` function raises ``AssertionError`` when the oracle disagrees with a value
worked by hand, a closed form, an exact small-integer case, or a brute-force scalar loop.
They read the oracle through its module attributes at call time, so a test can plant a
mistake in the oracle (monkeypatch) and check that some pin catches it.
"""
from __future__ import annotations

import json
import math
import pathlib

import numpy as np

import oracle.mamba2 as m2

GOLDEN = pathlib.Path(__file__).parent / "golden"


def _rng(seed):
    return np.random.default_rng(seed)


def _tiny_inputs(seed, bsz=2, k=6, H=2, G=1, P=2, N=3):
    r = _rng(seed)
    xs = r.standard_normal((bsz, k, H, P))
    Bs = r.standard_normal((bsz, k, G, N)) / np.sqrt(N)
    Cs = r.standard_normal((bsz, k, G, N)) / np.sqrt(N)
    dts = np.log1p(np.exp(r.standard_normal((bsz, k, H)) - 2.0))
    A = -np.exp(r.uniform(0, np.log(16.0), H))
    D = r.standard_normal(H)
    h0 = 0.1 * r.standard_normal((bsz, H, P, N))
    return xs, Bs, Cs, dts, A, D, h0


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ---------------------------------------------------------------- hand-worked values
def pin_golden_recurrence():
    """Decoder outputs and states equal values worked on paper."""
    doc = json.loads((GOLDEN / "recurrence_hand_worked.json").read_text())
    for case in doc["cases"]:
        A = np.array([-math.log(2.0) if a == "-ln2" else float(a) for a in case["A"]])
        D = np.array(case["D"], dtype=np.float64)
        H, P, N = case["nheads"], case["headdim"], case["dstate"]
        dec = m2.Mamba2Decoder(A, D, case["ngroups"], np.zeros((1, H, P, N)))
        for st in case["steps"]:
            y = dec.step(np.array([st["x"]], float), np.array([st["B"]], float),
                         np.array([st["C"]], float), np.array([st["dt"]], float))
            assert np.allclose(y[0], np.array(st["y"], float), rtol=1e-14, atol=1e-14), \
                (case["name"], y[0], st["y"])
            assert np.allclose(dec.h[0], np.array(st["h"], float), rtol=1e-14, atol=1e-14), \
                (case["name"], dec.h[0], st["h"])


# ---------------------------------------------------------------- brute force
def pin_brute_force_scalar_loops():
    """The vectorised step equals the definition written as scalar Python loops."""
    xs, Bs, Cs, dts, A, D, h0 = _tiny_inputs(11, bsz=2, k=5, H=4, G=2, P=2, N=3)
    bsz, k, H, P = xs.shape
    G, N = Bs.shape[2], Bs.shape[3]
    dec = m2.Mamba2Decoder(A, D, G, h0)
    h = [[[[float(h0[b, hh, p, n]) for n in range(N)] for p in range(P)]
          for hh in range(H)] for b in range(bsz)]
    for t in range(k):
        y = dec.step(xs[:, t], Bs[:, t], Cs[:, t], dts[:, t])
        for b in range(bsz):
            for hh in range(H):
                g = hh // (H // G)
                a = math.exp(dts[b, t, hh] * A[hh])
                for p in range(P):
                    acc = 0.0
                    for n in range(N):
                        h[b][hh][p][n] = a * h[b][hh][p][n] + dts[b, t, hh] * xs[b, t, hh, p] * Bs[b, t, g, n]
                        acc += h[b][hh][p][n] * Cs[b, t, g, n]
                    ref = acc + D[hh] * xs[b, t, hh, p]
                    assert abs(y[b, hh, p] - ref) <= 1e-12 * (1 + abs(ref)), (t, b, hh, p)
    assert _rel(dec.h, np.array(h)) < 1e-12


# ---------------------------------------------------------------- exact cases
def pin_integer_outer_product_sum():
    """A = 0, dt = 1: the state is exactly sum_s x_s B_s^T and y = h C + D x, exact in
    FP64 for small integers (checked bit for bit against integer arithmetic)."""
    r = _rng(3)
    bsz, k, H, G, P, N = 2, 7, 4, 2, 3, 5
    xi = r.integers(-8, 9, (bsz, k, H, P))
    Bi = r.integers(-8, 9, (bsz, k, G, N))
    Ci = r.integers(-8, 9, (bsz, k, G, N))
    Di = r.integers(-4, 5, H)
    dec = m2.Mamba2Decoder(np.zeros(H), Di.astype(float), G, np.zeros((bsz, H, P, N)))
    acc = np.zeros((bsz, H, P, N), dtype=np.int64)
    for t in range(k):
        y = dec.step(xi[:, t].astype(float), Bi[:, t].astype(float), Ci[:, t].astype(float),
                     np.ones((bsz, H)))
        for hh in range(H):
            g = hh // (H // G)
            acc[:, hh] += xi[:, t, hh, :, None] * Bi[:, t, g, None, :]
        yi = np.zeros((bsz, H, P), dtype=np.int64)
        for hh in range(H):
            g = hh // (H // G)
            yi[:, hh] = (acc[:, hh] * Ci[:, t, g, None, :]).sum(-1) + Di[hh] * xi[:, t, hh]
        assert np.array_equal(dec.h, acc.astype(float))
        assert np.array_equal(y, yi.astype(float))


def pin_zero_input_pure_decay():
    """x = 0: h_k = exp(A * sum_r dt_r) * h0 (pure decay); dt = 0: the state is kept."""
    xs, Bs, Cs, dts, A, D, h0 = _tiny_inputs(5, k=6)
    dec = m2.Mamba2Decoder(A, D, Bs.shape[2], h0)
    for t in range(xs.shape[1]):
        y = dec.step(np.zeros_like(xs[:, t]), Bs[:, t], Cs[:, t], dts[:, t])
        Gam = np.exp(A[None, :] * dts[:, : t + 1].sum(axis=1))
        assert _rel(dec.h, Gam[:, :, None, None] * h0) < 1e-13
        yref = np.einsum("bhpn,bn->bhp", Gam[:, :, None, None] * h0, Cs[:, t, 0])
        assert _rel(y, yref) < 1e-13
    dec = m2.Mamba2Decoder(A, D, Bs.shape[2], h0)
    y = dec.step(xs[:, 0], Bs[:, 0], Cs[:, 0], np.zeros_like(dts[:, 0]))
    assert np.array_equal(dec.h, h0)
    assert _rel(y, np.einsum("bhpn,bn->bhp", h0, Cs[:, 0, 0]) + D[None, :, None] * xs[:, 0]) < 1e-14


def pin_zero_state_single_update():
    """One update from a zero state: (dt x B^T) C = dt (B . C) x, plus the D x skip."""
    xs, Bs, Cs, dts, A, D, h0 = _tiny_inputs(7, k=1, H=4, G=2)
    dec = m2.Mamba2Decoder(A, D, 2, np.zeros_like(h0))
    y = dec.step(xs[:, 0], Bs[:, 0], Cs[:, 0], dts[:, 0])
    for hh in range(4):
        g = hh // 2
        bc = np.sum(Bs[:, 0, g] * Cs[:, 0, g], axis=-1)
        ref = (dts[:, 0, hh] * bc)[:, None] * xs[:, 0, hh] + D[hh] * xs[:, 0, hh]
        assert _rel(y[:, hh], ref) < 1e-14


# ---------------------------------------------------------------- closed forms
def pin_window_closed_form():
    """The unrolled window (checkpoint + records) equals the step recurrence, to 1e-12."""
    xs, Bs, Cs, dts, A, D, h0 = _tiny_inputs(1, bsz=3, k=8, H=4, G=2, P=2, N=3)
    dec = m2.Mamba2Decoder(A, D, 2, h0)
    for k in range(1, xs.shape[1] + 1):
        y = dec.step(xs[:, k - 1], Bs[:, k - 1], Cs[:, k - 1], dts[:, k - 1])
        hk = m2.window_state(h0, xs[:, :k], Bs[:, :k], dts[:, :k], A)
        yk = m2.window_output(h0, xs[:, :k], Bs[:, :k], dts[:, :k], Cs[:, k - 1], A, D)
        assert _rel(hk, dec.h) < 1e-12, k
        assert _rel(yk, y) < 1e-12, k


def pin_window_length_invariance():
    """Replay with any window L (outputs from checkpoint + buffer, fold every L records)
    gives the recurrence's outputs; L = 1 is the conventional step."""
    xs, Bs, Cs, dts, A, D, h0 = _tiny_inputs(2, bsz=2, k=17, H=2, G=1, P=3, N=2)
    ref = m2.Mamba2Decoder(A, D, 1, h0)
    yref = [ref.step(xs[:, t], Bs[:, t], Cs[:, t], dts[:, t]) for t in range(xs.shape[1])]
    for L in (1, 2, 3, 4, 8, 16):
        ckpt, first = h0.copy(), 0
        for t in range(xs.shape[1]):
            sl = slice(first, t + 1)
            y = m2.window_output(ckpt, xs[:, sl], Bs[:, sl], dts[:, sl], Cs[:, t], A, D)
            assert _rel(y, yref[t]) < 1e-12, (L, t)
            if t + 1 - first == L:
                ckpt, first = m2.window_state(ckpt, xs[:, sl], Bs[:, sl], dts[:, sl], A), t + 1


def pin_draft_matrix_form():
    """Output-only evaluation of T drafts against n records equals decoding the records,
    then each draft in turn."""
    for n in (0, 1, 5):
        xs, Bs, Cs, dts, A, D, h0 = _tiny_inputs(20 + n, bsz=2, k=n + 4, H=4, G=2, P=3, N=2)
        T = 4
        dec = m2.Mamba2Decoder(A, D, 2, h0)
        for t in range(n):
            dec.step(xs[:, t], Bs[:, t], Cs[:, t], dts[:, t])
        want = dec.verify(xs[:, n:], Bs[:, n:], Cs[:, n:], dts[:, n:])
        got = m2.draft_outputs(h0, (xs[:, :n], Bs[:, :n], dts[:, :n]),
                               (xs[:, n:], Bs[:, n:], Cs[:, n:], dts[:, n:]), A, D)
        assert got.shape == (2, T, 4, 3)
        assert _rel(got, want) < 1e-12, n


# ---------------------------------------------------------------- speculative rollback
def pin_verify_then_truncate():
    """Verify T drafts then commit a of them == decode only the accepted prefix."""
    xs, Bs, Cs, dts, A, D, h0 = _tiny_inputs(9, bsz=5, k=4, H=2, G=1)
    accept = np.array([0, 1, 2, 3, 4])
    dec = m2.Mamba2Decoder(A, D, 1, h0)
    ys = dec.verify(xs, Bs, Cs, dts)
    assert np.array_equal(dec.h, h0)            # verify keeps the committed state
    dec.commit(accept, xs, Bs, dts)
    for b in range(5):
        one = m2.Mamba2Decoder(A, D, 1, h0[b:b + 1])
        for j in range(4):
            y = one.step(xs[b:b + 1, j], Bs[b:b + 1, j], Cs[b:b + 1, j], dts[b:b + 1, j])
            assert _rel(ys[b:b + 1, j], y) < 1e-14
            if j + 1 == accept[b]:
                break
        if accept[b] == 0:
            one.h = h0[b:b + 1]
        assert _rel(dec.h[b:b + 1], one.h) < 1e-14, b


ALL_PINS = [
    pin_golden_recurrence, pin_brute_force_scalar_loops, pin_integer_outer_product_sum,
    pin_zero_input_pure_decay, pin_zero_state_single_update, pin_window_closed_form,
    pin_window_length_invariance, pin_draft_matrix_form, pin_verify_then_truncate,
]


def pin_window_rounding_only_at_window_ends():
    """The periodic low-precision checkpoint: with an identity rounding the decoder is the
    plain one; a rounding is applied exactly once per window, after the window's last step,
    and that step's output is read before it."""
    xs, Bs, Cs, dts, A, D, h0 = _tiny_inputs(30, bsz=2, k=10, H=2, G=1, P=2, N=3)
    calls = []

    def count(h):
        calls.append(1)
        return h

    plain = m2.Mamba2Decoder(A, D, 1, h0)
    counted = m2.Mamba2Decoder(A, D, 1, h0, window_round=count, window_L=4)
    zeroing = m2.Mamba2Decoder(A, D, 1, h0, window_round=np.zeros_like, window_L=4)
    for t in range(10):
        args = (xs[:, t], Bs[:, t], Cs[:, t], dts[:, t])
        y0, y1, y2 = plain.step(*args), counted.step(*args), zeroing.step(*args)
        assert np.array_equal(y0, y1)
        if t < 4:
            assert np.array_equal(y0, y2)
        if t == 3:
            assert np.array_equal(zeroing.h, np.zeros_like(h0))
    assert len(calls) == 2
    assert np.array_equal(plain.h, counted.h)


ALL_PINS.append(pin_window_rounding_only_at_window_ends)
