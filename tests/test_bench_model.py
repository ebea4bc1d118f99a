"""The benchmark's algorithmic-byte model, against what the method fixes.

Source: "ReplaySSM: Rethinking State Storage for Faster Hybrid-Model Decoding", "Benefit 1:
Reduce state memory traffic": over a window of L tokens the conventional step reads and
writes the state L times each, ReplaySSM reads it L times and writes it once, so the state
traffic ratio is (L + 1) / (2L); a non-flush step writes only the new record (x, B, dt).
These relations pin bench.py's per-call byte counts, from which every roofline figure is
computed. (Host-side: no GPU needed.)
"""
import sys
from pathlib import Path

import pytest

sys.path.insert(0, str(Path(__file__).resolve().parent.parent))
import bench  # noqa: E402

W = bench.WORKLOAD
S = W["batch"] * W["nheads"] * W["headdim"] * W["dstate"]  # state elements


def test_record_is_x_B_dt_of_a_token():
    # x: H x P per sequence, B: G x N (per group), dt: H; bf16 inputs
    assert bench.record_bytes(W, 2) == (128 * 64 + 8 * 128 + 128) * 2 == 18688


def test_non_flush_step_reads_state_and_records_and_writes_one_record():
    rec = W["batch"] * bench.record_bytes(W, 2)
    base = bench.step_bytes(W, 0, False)
    for n in (1, 7, 15):
        assert bench.step_bytes(W, n, False) - base == n * rec
    inputs = W["batch"] * (W["nheads"] * W["headdim"] + 2 * W["ngroups"] * W["dstate"] + W["nheads"]) * 2
    y = W["batch"] * W["nheads"] * W["headdim"] * 4
    assert base == S * 4 + inputs + y + rec


def test_flush_writes_the_state_once_and_no_record():
    rec = W["batch"] * bench.record_bytes(W, 2)
    for n in (3, 15):
        assert bench.step_bytes(W, n, True) - bench.step_bytes(W, n, False) == S * 4 - rec


def test_window_state_traffic_ratio_is_l_plus_one_over_two_l():
    L = W["L"]
    inputs = W["batch"] * (W["nheads"] * W["headdim"] + 2 * W["ngroups"] * W["dstate"] + W["nheads"]) * 2
    y = W["batch"] * W["nheads"] * W["headdim"] * 4
    rec = W["batch"] * bench.record_bytes(W, 2)
    # the conventional step: the state read and written, plus the token's inputs and y
    assert bench.conv_bytes(W) == 2 * S * 4 + inputs + y
    window = sum(bench.step_bytes(W, t, t == L - 1) for t in range(L))
    records = sum(range(L)) * rec + (L - 1) * rec   # buffered records read + records appended
    state = window - records - L * (inputs + y)
    assert state == (L + 1) * S * 4
    assert state / (L * 2 * S * 4) == pytest.approx((L + 1) / (2 * L))


def test_read_copies_change_only_the_state_bytes():
    for fmt, (rcb, slab_scale) in bench.RC_BYTES.items():
        copy = S * rcb + (W["batch"] * W["nheads"] * 4 if slab_scale else 0)
        nf = bench.step_bytes(W, 5, False, rc_bytes=rcb, slab_scale=slab_scale)
        assert nf - bench.step_bytes(W, 5, False) == pytest.approx(copy - S * 4), fmt
        fl = bench.step_bytes(W, 15, True, rc_bytes=rcb, slab_scale=slab_scale)
        assert fl - bench.step_bytes(W, 15, True) == pytest.approx(copy), fmt   # the copy written too
        shared = bench.step_bytes(W, 15, True, rc_bytes=rcb, shared=True, slab_scale=slab_scale)
        assert shared - (fl - 2 * S * 4 - copy) == pytest.approx(2 * copy), fmt  # the copy read and written
