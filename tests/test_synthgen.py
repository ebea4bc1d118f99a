"""The seeded input generator: determinism, subset independence, distributions (CPU)."""
import numpy as np

import synthgen as sg


def test_counter_based_subsets_match_full_draw():
    shape = sg.LayerShape(6, 4, 8, 16, 2, "bf16")
    full = sg.token_inputs(shape, 0, np.arange(5))
    part = sg.token_inputs(shape, 0, [3], seqs=[4, 1])
    for k in ("x", "B", "C", "dt"):
        assert np.array_equal(part[k].store, full[k].store[[4, 1]][:, [3]])
    small = sg.token_inputs(sg.LayerShape(2, 4, 8, 16, 2, "bf16"), 0, np.arange(5))
    assert np.array_equal(small["x"].store, full["x"].store[:2])     # batch-size invariant


def test_seeds_and_streams_differ():
    a = sg.normal(0, 1, np.arange(1000))
    assert not np.allclose(a, sg.normal(1, 1, np.arange(1000)))
    assert not np.allclose(a, sg.normal(0, 2, np.arange(1000)))


def test_distributions():
    shape = sg.LayerShape(8, 8, 64, 128, 2, "f32")
    d = sg.token_inputs(shape, 0, np.arange(8))
    x, B, dt = d["x"].f64, d["B"].f64, d["dt"].f64
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
    assert abs(B.std() * np.sqrt(128) - 1) < 0.05
    assert dt.min() > 0 and abs(np.median(dt) - np.log1p(np.exp(-2.0))) < 0.02
    A, D = sg.head_params(64, 0)
    assert np.all(A <= -1) and np.all(A >= -16) and A.dtype == np.float32
    u = sg.uniform(3, 9, np.arange(100000))
    assert u.min() > 0 and u.max() < 1 and abs(u.mean() - 0.5) < 0.01


def test_bf16_storage_is_rounded_and_widened_exactly():
    shape = sg.LayerShape(2, 2, 8, 16, 1, "bf16")
    d = sg.token_inputs(shape, 0, [0])
    assert d["x"].store.dtype == np.uint16
    back = (d["x"].store.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(back, d["x"].f64)


def test_accept_lengths_cover_range():
    a = np.concatenate([sg.accept_lengths(512, 4, 0, c) for c in range(8)])
    assert a.min() == 0 and a.max() == 4 and a.dtype == np.int32
    assert set(np.unique(a)) == {0, 1, 2, 3, 4}
