"""The decode step for callers that must not allocate device memory.

Some callers cannot allocate when they decode (an engine plugin given only its buffers,
memory pre-claimed by another framework's pool, code under stream capture). For them,
replay_step_static_scratch keeps replay_step's per-step scratch -- arrival counters, plan,
record coefficients -- in a fixed array inside the library. These tests call it through the C ABI and
check it against replay_step on identical stores, call after call. This file is collected
last on purpose, so a failing run has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synthgen as sg
from gpu_util import make_store, rel_vec_err, step_inputs
from hybrid_model_ssm_mamba_gb300 import replay as R

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _c_call(lib, store, devs, y):
    ptrs = [t.data_ptr() for t in devs]
    stream = torch.cuda.current_stream().cuda_stream
    return lib.replay_step_static_scratch(store.handle, *ptrs, y.data_ptr(), stream)


def test_matches_replay_step_on_consecutive_calls(lib):
    """Two stores fed the same tokens: one through replay_step, one through the static-scratch
    entry point. Outputs, checkpoints and ring pointers agree on every call, across a flush."""
    shape = sg.LayerShape(5, 8, 64, 128, 2, "bf16")
    ref, _, _ = make_store(shape, 31, L=3)
    new, _, _ = make_store(shape, 31, L=3)
    y_ref = torch.empty(5, 8, 64, device="cuda")
    y_new = torch.empty_like(y_ref)
    for t in range(5):                      # two calls in a row, then through a flush and on
        devs, _ = step_inputs(shape, 31, t)
        ref.step(*devs, y_ref)
        assert _c_call(lib, new, devs, y_new) == 0
        torch.cuda.synchronize()
        assert rel_vec_err(y_new.cpu().numpy(), y_ref.cpu().numpy(), 2).max() <= TOL, t
        assert torch.equal(new.region("meta"), ref.region("meta")), t
    assert rel_vec_err(new.region("h0").cpu().numpy(), ref.region("h0").cpu().numpy(), 2).max() <= TOL
    assert new.status() == 0 and ref.status() == 0


def test_rejects_more_coefficients_than_the_array_holds(lib):
    shape = sg.LayerShape(128, 128, 64, 64, 1, "bf16")      # 128 * 128 * 65 > 2**20
    st, _, _ = make_store(shape, 33, L=64)
    assert shape.batch * shape.nheads * (st.layout.cap + 1) > R.REPLAY_STATIC_MAX_COEFS
    devs, _ = step_inputs(shape, 33, 0)
    y = torch.zeros(128, 128, 64, device="cuda")
    assert _c_call(lib, st, devs, y) == -3
    torch.cuda.synchronize()
    assert not torch.any(y != 0)


def test_rejects_batch_beyond_the_limit(lib):
    limit = R.REPLAY_STATIC_MAX_BATCH
    shape = sg.LayerShape(limit + 1, 1, 64, 64, 1, "f32")
    st, _, _ = make_store(shape, 32, L=2)
    devs, _ = step_inputs(shape, 32, 0)
    y = torch.zeros(limit + 1, 1, 64, device="cuda")
    meta_before = st.region("meta").clone()
    assert _c_call(lib, st, devs, y) == -3            # REPLAY_ECAPACITY, nothing launched
    torch.cuda.synchronize()
    assert not torch.any(y != 0)
    assert torch.equal(st.region("meta"), meta_before)
