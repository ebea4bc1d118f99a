"""GPU parity of the conventional baselines (load-update-store step, snapshot-per-draft
verify) against the FP64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import synthgen as sg
from gpu_util import draft_device, make_cfg, rel_vec_err, step_inputs
from hybrid_model_ssm_mamba_gb300 import replay as R
from oracle.mamba2 import Mamba2Decoder

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _params(shape, seed):
    A, D = sg.head_params(shape.nheads, seed)
    return torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda(), A.astype(float), D.astype(float)


@pytest.mark.parametrize("N,dtype", [(128, "f32"), (128, "bf16"), (64, "bf16"), (256, "f32")])
def test_conv_step_fp32_state(N, dtype):
    shape = sg.LayerShape(3, 8, 64, N, 2, dtype)
    cfg = make_cfg(shape)
    Ad, Dd, A, D = _params(shape, 21)
    state = torch.zeros(3, 8, 64, N, device="cuda")
    orc = Mamba2Decoder(A, D, 2, np.zeros((3, 8, 64, N)))
    y = torch.empty(3, 8, 64, device="cuda")
    for t in range(30):
        devs, f64 = step_inputs(shape, 21, t)
        R.conv_step(cfg, state, R.REPLAY_F32, Ad, Dd, *devs, y)
        assert rel_vec_err(y.cpu().numpy(), orc.step(*f64), 2).max() <= TOL, t
    assert rel_vec_err(state.cpu().numpy(), orc.h, 2).max() <= TOL


def test_conv_step_bf16_state_drifts_more_than_fp32():
    """A bf16 stored state re-enters the recurrence every step (the pages' 'State
    quantization'); its error is larger than the FP32 path's but bounded here."""
    shape = sg.LayerShape(4, 8, 64, 128, 1, "f32")
    cfg = make_cfg(shape)
    Ad, Dd, A, D = _params(shape, 22)
    s16 = torch.zeros(4, 8, 64, 128, device="cuda", dtype=torch.bfloat16)
    s32 = torch.zeros(4, 8, 64, 128, device="cuda")
    orc = Mamba2Decoder(A, D, 1, np.zeros((4, 8, 64, 128)))
    y16 = torch.empty(4, 8, 64, device="cuda")
    y32 = torch.empty_like(y16)
    e16 = e32 = 0.0
    for t in range(64):
        devs, f64 = step_inputs(shape, 22, t)
        R.conv_step(cfg, s16, R.REPLAY_BF16, Ad, Dd, *devs, y16)
        R.conv_step(cfg, s32, R.REPLAY_F32, Ad, Dd, *devs, y32)
        yr = orc.step(*f64)
        e16 = max(e16, rel_vec_err(y16.cpu().numpy(), yr, 2).max())
        e32 = max(e32, rel_vec_err(y32.cpu().numpy(), yr, 2).max())
    assert e32 <= TOL and e16 > e32 and e16 < 0.1, (e16, e32)


def test_conv_verify_snapshot_and_commit():
    shape = sg.LayerShape(6, 4, 64, 128, 2, "bf16")
    T = 3
    cfg = make_cfg(shape, T=T)
    Ad, Dd, A, D = _params(shape, 23)
    snaps = torch.zeros(6, T + 1, 4, 64, 128, device="cuda")
    cur = torch.zeros(6, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    orc = Mamba2Decoder(A, D, 2, np.zeros((6, 4, 64, 128)))
    y = torch.empty(6, T, 4, 64, device="cuda")
    for call in range(10):
        devs, f64 = draft_device(shape, 23, call, T)
        R.conv_verify_snapshot(cfg, T, snaps, cur, Ad, Dd, *devs, y)
        assert rel_vec_err(y.cpu().numpy(), orc.verify(*f64), 3).max() <= TOL, call
        acc = sg.accept_lengths(6, T, 23, call)
        R.conv_commit(6, T, cur, torch.from_numpy(acc).cuda(), status)
        orc.commit(acc, f64[0], f64[1], f64[3])
        c = cur.cpu().numpy()
        cur_state = snaps.cpu().numpy()[np.arange(6), c]
        assert rel_vec_err(cur_state, orc.h, 2).max() <= TOL, call
    assert status.item() == 0
    R.conv_commit(6, T, cur, torch.full((6,), T + 1, dtype=torch.int32, device="cuda"), status)
    assert status.item() == R.REPLAY_DEV_BAD_ACCEPT
