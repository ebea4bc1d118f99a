"""Helpers of the GPU parity tests: seeded inputs on the device, the oracle beside them,
and the error metric.

Error metric: per output vector (sequence, head, token) the relative infinity-norm error
||y - y*||_inf / ||y*||_inf; per state slab the same over its P x N values.
"""
from __future__ import annotations

import numpy as np
import torch

import synthgen as sg
from hybrid_model_ssm_mamba_gb300 import replay as R

DTYPE = {"f32": R.REPLAY_F32, "bf16": R.REPLAY_BF16}


def dev(drawn, dtype: str, device="cuda") -> torch.Tensor:
    """A drawn input as the device tensor the library consumes."""
    a = np.ascontiguousarray(drawn.store)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def rel_vec_err(y, yref, axis_from: int) -> np.ndarray:
    """Relative inf-norm error per vector; the vector spans axes ``axis_from..``."""
    y = np.asarray(y, dtype=np.float64)
    yref = np.asarray(yref, dtype=np.float64)
    ax = tuple(range(axis_from, y.ndim))
    num = np.max(np.abs(y - yref), axis=ax)
    den = np.max(np.abs(yref), axis=ax)
    return num / np.maximum(den, 1e-30)


def make_cfg(shape: sg.LayerShape, L=16, T=0, read_copy=R.REPLAY_RC_NONE) -> R.ReplayConfig:
    return R.ReplayConfig(shape.batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups,
                          L, T, DTYPE[shape.dtype], read_copy)


def make_store(shape: sg.LayerShape, seed=0, L=16, T=0, read_copy=R.REPLAY_RC_NONE):
    A, D = sg.head_params(shape.nheads, seed)
    st = R.ReplayStore(make_cfg(shape, L, T, read_copy), torch.from_numpy(A), torch.from_numpy(D))
    return st, A.astype(np.float64), D.astype(np.float64)


def step_inputs(shape, seed, t, seqs=None):
    """Device tensors of token t (all sequences) and the FP64 values of sequences `seqs`."""
    d = sg.token_inputs(shape, seed, [t])
    devs = [dev(_slice_t(d[k]), shape.dtype) for k in ("x", "B", "C", "dt")]
    sel = slice(None) if seqs is None else seqs
    f64 = [d[k].f64[sel, 0] for k in ("x", "B", "C", "dt")]
    return devs, f64


class _View:
    def __init__(self, store, f64):
        self.store, self.f64 = store, f64


def _slice_t(drawn):
    return _View(np.ascontiguousarray(drawn.store[:, 0]), drawn.f64[:, 0])


def draft_device(shape, seed, call, T):
    d = sg.draft_inputs(shape, seed, call, T)
    devs = [dev(d[k], shape.dtype) for k in ("x", "B", "C", "dt")]
    f64 = [d[k].f64 for k in ("x", "B", "C", "dt")]
    return devs, f64
