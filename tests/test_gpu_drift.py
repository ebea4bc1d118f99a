"""Dual-precision drift over a long decode (GPU vs the FP64 oracle).

The tiny layer's shape at batch 256 decodes 4096 tokens ten ways on identical inputs:
ReplaySSM with the FP32 checkpoint only, with a bf16, E4M3 or NVFP4 read copy, with a
shared bf16, E4M3, FP16 (stochastically rounded) or NVFP4 checkpoint (the copy is the
recurrence state, rounded once per window and fed back), with an FP16 stochastically
rounded checkpoint beside an NVFP4 read copy, and the conventional step with a bf16 stored
state. The oracle follows four seeded sequences. Source: "ReplaySSM: Rethinking State Storage for Faster Hybrid-Model Decoding",
sections "State quantization" (a low-precision state's rounding re-enters the recurrence
every step) and "Benefit 3" (a read copy's error stays within a window and does not grow).

Checked: the FP32 path stays within 1e-4 throughout; the bf16 copy within 1e-2; the read
copies' error does not grow with length (last quarter vs first quarter). Reported: the
per-512-token max / mean of the per-vector relative error for all ten paths (in the run's
closing summary, and as JSON in $REPLAY_DRIFT_REPORT when that is set).
"""
import json
import os

import numpy as np
import pytest
import torch

import synthgen as sg
from gpu_util import dev, make_cfg, make_store, rel_vec_err
from hybrid_model_ssm_mamba_gb300 import replay as R
from oracle.mamba2 import Mamba2Decoder

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def test_dual_precision_drift_4096_tokens(report):
    steps, L, seed, chunk = 4096, 16, 41, 512
    shape = sg.LayerShape(256, 8, 64, 128, 1, "f32")
    sel = np.array([3, 100, 171, 250])
    stores = {name: make_store(shape, seed, L=L, read_copy=rc)[0] for name, rc in
              (("replay_fp32", R.REPLAY_RC_NONE), ("replay_bf16_copy", R.REPLAY_RC_BF16),
               ("replay_e4m3_copy", R.REPLAY_RC_FP8E4M3))}
    A, D = sg.head_params(shape.nheads, seed)
    for name, rc, shared, fmt in (
            ("shared_bf16_checkpoint", R.REPLAY_RC_BF16, 1, 0), ("shared_e4m3_checkpoint", R.REPLAY_RC_FP8E4M3, 1, 0),
            ("shared_fp16_sr_checkpoint", R.REPLAY_RC_FP16, 1, 0), ("replay_nvfp4_copy", R.REPLAY_RC_NVFP4, 0, 0),
            ("shared_nvfp4_checkpoint", R.REPLAY_RC_NVFP4, 1, 0),
            ("fp16_sr_checkpoint_nvfp4_copy", R.REPLAY_RC_NVFP4, 0, R.REPLAY_CKPT_F16_SR)):
        cfg_s = R.ReplayConfig(256, 8, 64, 128, 1, L, 0, R.REPLAY_F32, rc, shared, fmt)
        stores[name] = R.ReplayStore(cfg_s, torch.from_numpy(A), torch.from_numpy(D))
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    cfg = make_cfg(shape, L=L)
    state16 = torch.zeros(256, 8, 64, 128, device="cuda", dtype=torch.bfloat16)
    orc = Mamba2Decoder(A.astype(np.float64), D.astype(np.float64), 1, np.zeros((4, 8, 64, 128)))
    names = list(stores) + ["conv_bf16_state"]
    ys = {n: torch.empty(256, 8, 64, device="cuda") for n in names}
    err = {n: np.zeros(steps) for n in names}
    mean = {n: np.zeros(steps) for n in names}
    for t0 in range(0, steps, 64):
        d = sg.token_inputs(shape, seed, np.arange(t0, t0 + 64))
        for i in range(64):
            t = t0 + i
            devs = [dev(_at(d[k], i), "f32") for k in ("x", "B", "C", "dt")]
            for n, st in stores.items():
                st.step(*devs, ys[n])
            R.conv_step(cfg, state16, R.REPLAY_BF16, Ad, Dd, *devs, ys["conv_bf16_state"])
            yref = orc.step(*(d[k].f64[sel, i] for k in ("x", "B", "C", "dt")))
            for n in names:
                e = rel_vec_err(ys[n][sel].cpu().numpy(), yref, 2)
                err[n][t], mean[n][t] = e.max(), e.mean()
    table = {n: {"max_per_512": [float(err[n][i:i + chunk].max()) for i in range(0, steps, chunk)],
                  "mean_per_512": [float(mean[n][i:i + chunk].mean()) for i in range(0, steps, chunk)]}
              for n in names}
    print(json.dumps(table))
    report("drift over 4096 tokens (tiny-layer shape, batch 256, L 16; per-vector relative error of y "
           "vs the FP64 oracle on 4 sequences), max / mean per 512 tokens:")
    for n in names:
        mx = " ".join(f"{v:.1e}" for v in table[n]["max_per_512"])
        mn = " ".join(f"{v:.1e}" for v in table[n]["mean_per_512"])
        report(f"  {n:32s} max {mx} | mean {mn}")
    if os.environ.get("REPLAY_DRIFT_REPORT"):
        with open(os.environ["REPLAY_DRIFT_REPORT"], "w") as f:
            json.dump({"workload": "tiny-layer shape, batch 256, 4096 tokens, L 16, oracle on 4 sequences",
                       "metric": "per-vector relative inf-norm error of y vs the FP64 oracle",
                       "paths": table}, f, indent=1)
    assert err["replay_fp32"].max() <= 1e-4
    assert err["replay_bf16_copy"].max() <= 1e-2
    for n in ("replay_bf16_copy", "replay_e4m3_copy", "replay_nvfp4_copy", "fp16_sr_checkpoint_nvfp4_copy"):
        q = steps // 4
        assert mean[n][-q:].mean() <= 2.0 * mean[n][:q].mean() + 1e-6, n   # the read error does not grow
    for st in stores.values():
        assert st.status() == 0


class _At:
    def __init__(self, store, f64):
        self.store, self.f64 = store, f64


def _at(drawn, i):
    return _At(np.ascontiguousarray(drawn.store[:, i]), drawn.f64[:, i])


def test_shared_checkpoint_error_accumulates_with_slow_decay(report):
    """With heads whose decay is slow (A scaled by 1e-3, so a window keeps ~99.8 % of the
    state), a shared bf16 checkpoint's rounding error is fed back every window and adds up,
    while a bf16 read copy's error stays a read error. Source: the post's section "Benefit 3"
    (a shared low-precision checkpoint accumulates error with length; keeping the recurrence
    in FP32 removes the growth). Reported per 256 tokens; checked: the read copy's error does
    not grow, and at the end the shared checkpoint's error is the larger."""
    steps, L, seed, chunk = 2048, 16, 43, 256
    shape = sg.LayerShape(64, 8, 64, 128, 1, "f32")
    sel = np.array([1, 33])
    A, D = sg.head_params(shape.nheads, seed)
    A = (A * np.float32(1e-3)).astype(np.float32)
    stores = {}
    for name, shared in (("bf16_read_copy", 0), ("shared_bf16_checkpoint", 1)):
        cfg = R.ReplayConfig(64, 8, 64, 128, 1, L, 0, R.REPLAY_F32, R.REPLAY_RC_BF16, shared)
        stores[name] = R.ReplayStore(cfg, torch.from_numpy(A), torch.from_numpy(D))
    orc = Mamba2Decoder(A.astype(np.float64), D.astype(np.float64), 1, np.zeros((2, 8, 64, 128)))
    y = {n: torch.empty(64, 8, 64, device="cuda") for n in stores}
    mean = {n: np.zeros(steps) for n in stores}
    for t0 in range(0, steps, 64):
        d = sg.token_inputs(shape, seed, np.arange(t0, t0 + 64))
        for i in range(64):
            devs = [dev(_at(d[k], i), "f32") for k in ("x", "B", "C", "dt")]
            for n, st in stores.items():
                st.step(*devs, y[n])
            yref = orc.step(*(d[k].f64[sel, i] for k in ("x", "B", "C", "dt")))
            for n in stores:
                mean[n][t0 + i] = rel_vec_err(y[n][sel].cpu().numpy(), yref, 2).mean()
    table = {n: [float(mean[n][i:i + chunk].mean()) for i in range(0, steps, chunk)] for n in stores}
    print(json.dumps({"slow_decay_mean_per_256": table}))
    report("slow-decay heads (A x 1e-3, batch 64, 2048 tokens): mean error per 256 tokens:")
    for n, v in table.items():
        report(f"  {n:32s} " + " ".join(f"{e:.1e}" for e in v))
    q = steps // 4
    sep, shr = mean["bf16_read_copy"], mean["shared_bf16_checkpoint"]
    assert sep[-q:].mean() <= 2.0 * sep[q:2 * q].mean() + 1e-9
    assert shr[-q:].mean() > sep[-q:].mean()
    for st in stores.values():
        assert st.status() == 0
