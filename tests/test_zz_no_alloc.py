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
from oracle.mamba2 import Mamba2Decoder

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


@pytest.mark.parametrize("rc,bound", [(R.REPLAY_RC_NONE, TOL), (R.REPLAY_RC_BF16, 1e-2)])
def test_large_calls_through_the_prep_kernel(lib, rc, bound):
    """Calls of more than 1024 (sequence, head) slabs run a per-group prep kernel whose plan
    and record coefficients live in the array (16 x 128 heads, 8 groups, bf16 inputs). With a
    read copy the prep also appends the token's B and dt records. Three stores take the same
    tokens through two flushes: one by replay_step, one by this entry point, one alternating
    the two. Outputs, ring pointers and checkpoints agree; the oracle follows three sequences
    (within 1e-4, or the bf16 copy's 1e-2 for outputs read from the copy)."""
    shape = sg.LayerShape(16, 128, 64, 128, 8, "bf16")
    L, seed, sel = 4, 34, np.array([0, 7, 15])
    ref, A, D = make_store(shape, seed, L=L, read_copy=rc)
    new, _, _ = make_store(shape, seed, L=L, read_copy=rc)
    mix, _, _ = make_store(shape, seed, L=L, read_copy=rc)
    assert shape.batch * shape.nheads > 1024
    orc = Mamba2Decoder(A, D, shape.ngroups, np.zeros((len(sel), 128, 64, 128)))
    ys = [torch.empty(16, 128, 64, device="cuda") for _ in range(3)]
    for t in range(10):
        devs, f64 = step_inputs(shape, seed, t, sel)
        ref.step(*devs, ys[0])
        assert _c_call(lib, new, devs, ys[1]) == 0
        if t % 2:
            mix.step(*devs, ys[2])
        else:
            assert _c_call(lib, mix, devs, ys[2]) == 0
        torch.cuda.synchronize()
        y_ref = ys[0].cpu().numpy()
        for y in ys[1:]:
            assert rel_vec_err(y.cpu().numpy(), y_ref, 2).max() <= TOL, t
        yo = orc.step(*f64)
        assert rel_vec_err(y_ref[sel], yo, 2).max() <= (TOL if (t + 1) % L == 0 else bound), t
        for st in (new, mix):
            assert torch.equal(st.region("meta"), ref.region("meta")), t
        if (t + 1) % L == 0:
            h_ref = ref.region("h0").cpu().numpy()
            assert rel_vec_err(h_ref[sel], orc.h, 2).max() <= TOL, t
            for st in (new, mix):
                assert rel_vec_err(st.region("h0").cpu().numpy(), h_ref, 2).max() <= TOL, t
                if rc != R.REPLAY_RC_NONE:
                    assert torch.equal(st.region("rc"), ref.region("rc")), t
    for st in (ref, new, mix):
        assert st.status() == 0


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
