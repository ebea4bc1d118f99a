"""Thin Python binding of the ReplaySSM C ABI (``include/replayssm.h``).

Argument marshalling only: every step of the decode path runs in the CUDA library
``lib/libreplayssm.so``. Functions keep the C names; tensors are passed as device
pointers, so callers own all device memory (PyTorch allocates it) and the current
PyTorch CUDA stream is used unless one is given. A non-zero return code raises
:class:`ReplayError`. There is no fallback: if the library is not built, or CUDA is not
available, calls fail.
"""
from __future__ import annotations

import ctypes
import pathlib
import re

import torch

from . import build as _build

__all__ = [
    "ReplayError", "ReplayConfig", "ReplayLayout", "load_library", "header_functions",
    "REPLAY_F32", "REPLAY_BF16", "REPLAY_RC_NONE", "REPLAY_RC_BF16", "REPLAY_RC_FP8E4M3", "REPLAY_RC_FP16",
    "REPLAY_RC_NVFP4", "REPLAY_CKPT_F32", "REPLAY_CKPT_F16_SR",
    "REPLAY_DEV_BAD_META", "REPLAY_DEV_BAD_ACCEPT", "REPLAY_DEV_COPY_TIMEOUT",
    "replay_layout_of", "replay_store_bytes", "replay_alloc", "replay_free", "replay_reset",
    "replay_load_state", "replay_export_state", "replay_step", "replay_verify",
    "replay_commit", "replay_flush", "replay_status", "conv_step", "conv_verify_snapshot",
    "conv_commit", "ReplayStore",
]

HEADER = pathlib.Path(__file__).resolve().parent.parent / "include" / "replayssm.h"

REPLAY_F32, REPLAY_BF16 = 0, 1
REPLAY_RC_NONE, REPLAY_RC_BF16, REPLAY_RC_FP8E4M3, REPLAY_RC_FP16, REPLAY_RC_NVFP4 = 0, 1, 2, 3, 4
REPLAY_CKPT_F32, REPLAY_CKPT_F16_SR = 0, 1
REPLAY_DEV_BAD_META, REPLAY_DEV_BAD_ACCEPT, REPLAY_DEV_COPY_TIMEOUT = 1, 2, 4
REPLAY_STATIC_MAX_BATCH = 4096
REPLAY_STATIC_MAX_COEFS = 1048576
_ERRORS = {-1: "bad argument", -2: "unsupported shape or dtype", -3: "capacity exceeded",
           -4: "CUDA error"}


class ReplayError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {_ERRORS.get(code, 'unknown error')} ({code})")
        self.code = code


class ReplayConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "batch", "nheads", "headdim", "dstate", "ngroups", "window_L", "max_draft_T",
        "in_dtype", "read_copy", "shared_checkpoint", "checkpoint_format")]

    def __init__(self, batch, nheads, headdim, dstate, ngroups, window_L=16, max_draft_T=0,
                 in_dtype=REPLAY_F32, read_copy=REPLAY_RC_NONE, shared_checkpoint=0,
                 checkpoint_format=0):
        super().__init__(batch, nheads, headdim, dstate, ngroups, window_L, max_draft_T,
                         in_dtype, read_copy, shared_checkpoint, checkpoint_format)

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class ReplayLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "h0", "rc", "scale", "bscale", "xbuf", "bbuf", "dtbuf", "meta", "arrive", "status", "plan", "coef",
        "total")] + \
        [("cap", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "replay_layout_of": [ctypes.POINTER(ReplayConfig), ctypes.POINTER(ReplayLayout)],
    "replay_store_bytes": [ctypes.POINTER(ReplayConfig), ctypes.POINTER(ctypes.c_size_t)],
    "replay_alloc": [ctypes.POINTER(ReplayConfig), _P, ctypes.c_size_t, _P, _P, _P, ctypes.POINTER(_P)],
    "replay_free": [_P],
    "replay_reset": [_P, _P, _P],
    "replay_load_state": [_P, _P, _P],
    "replay_export_state": [_P, _P, _P],
    "replay_step": [_P, _P, _P, _P, _P, _P, _P],
    "replay_step_static_scratch": [_P, _P, _P, _P, _P, _P, _P],
    "replay_verify": [_P, _I, _P, _P, _P, _P, _P, _P],
    "replay_commit": [_P, _P, _P],
    "replay_flush": [_P, _P],
    "replay_status": [_P, ctypes.POINTER(_I), _I, _P],
    "conv_step": [ctypes.POINTER(ReplayConfig), _P, _I, _P, _P, _P, _P, _P, _P, _P, _P],
    "conv_verify_snapshot": [ctypes.POINTER(ReplayConfig), _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "conv_commit": [_I, _I, _P, _P, _P, _P],
    "replay_strerror": [_I],
    "replay_abi_version": [],
}

_lib = None


def header_functions() -> list[str]:
    """Names of the functions declared in the C header."""
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)


def load_library(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load ``libreplayssm.so`` (building it in-tree first if asked and needed)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.lib_path()
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not path.exists():
        raise RuntimeError(f"the ReplaySSM CUDA library is not built ({path}); run the build step")
    lib = ctypes.CDLL(str(path))
    for name, argtypes in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = argtypes
        fn.restype = ctypes.c_char_p if name == "replay_strerror" else ctypes.c_int
    _lib = lib
    return lib


def _check(fn: str, rc: int):
    if rc != 0:
        raise ReplayError(fn, rc)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ------------------------------------------------------------------ C calls, same names
def replay_layout_of(cfg: ReplayConfig) -> ReplayLayout:
    out = ReplayLayout()
    _check("replay_layout_of", load_library().replay_layout_of(ctypes.byref(cfg), ctypes.byref(out)))
    return out


def replay_store_bytes(cfg: ReplayConfig) -> int:
    n = ctypes.c_size_t()
    _check("replay_store_bytes", load_library().replay_store_bytes(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def replay_alloc(cfg, workspace, workspace_bytes, A, D, stream=None) -> int:
    h = _P()
    _check("replay_alloc", load_library().replay_alloc(
        ctypes.byref(cfg), _ptr(workspace), workspace_bytes, _ptr(A), _ptr(D), _stream(stream),
        ctypes.byref(h)))
    return h.value


def replay_free(store: int):
    _check("replay_free", load_library().replay_free(store))


def replay_reset(store, seq_mask=None, stream=None):
    _check("replay_reset", load_library().replay_reset(store, _ptr(seq_mask), _stream(stream)))


def replay_load_state(store, h, stream=None):
    _check("replay_load_state", load_library().replay_load_state(store, _ptr(h), _stream(stream)))


def replay_export_state(store, h_out, stream=None):
    _check("replay_export_state", load_library().replay_export_state(store, _ptr(h_out), _stream(stream)))


def replay_step(store, x, B, C, dt, y, stream=None):
    _check("replay_step", load_library().replay_step(
        store, _ptr(x), _ptr(B), _ptr(C), _ptr(dt), _ptr(y), _stream(stream)))


def replay_verify(store, T, x, B, C, dt, y, stream=None):
    _check("replay_verify", load_library().replay_verify(
        store, T, _ptr(x), _ptr(B), _ptr(C), _ptr(dt), _ptr(y), _stream(stream)))


def replay_commit(store, accept, stream=None):
    _check("replay_commit", load_library().replay_commit(store, _ptr(accept), _stream(stream)))


def replay_flush(store, stream=None):
    _check("replay_flush", load_library().replay_flush(store, _stream(stream)))


def replay_step_static_scratch(store, x, B, C, dt, y, stream=None):
    """replay_step whose scratch (per-sequence arrival counters) lives in a fixed array in
    the library, for callers that must not allocate device memory; batch is limited to
    REPLAY_STATIC_MAX_BATCH."""
    _check("replay_step_static_scratch", load_library().replay_step_static_scratch(
        store, _ptr(x), _ptr(B), _ptr(C), _ptr(dt), _ptr(y), _stream(stream)))


def replay_status(store, clear=False, stream=None) -> int:
    v = _I()
    _check("replay_status", load_library().replay_status(store, ctypes.byref(v), int(clear), _stream(stream)))
    return v.value


def conv_step(cfg, state, state_dtype, A, D, x, B, C, dt, y, stream=None):
    _check("conv_step", load_library().conv_step(
        ctypes.byref(cfg), _ptr(state), state_dtype, _ptr(A), _ptr(D), _ptr(x), _ptr(B), _ptr(C),
        _ptr(dt), _ptr(y), _stream(stream)))


def conv_verify_snapshot(cfg, T, snaps, cur, A, D, x, B, C, dt, y, stream=None):
    _check("conv_verify_snapshot", load_library().conv_verify_snapshot(
        ctypes.byref(cfg), T, _ptr(snaps), _ptr(cur), _ptr(A), _ptr(D), _ptr(x), _ptr(B), _ptr(C),
        _ptr(dt), _ptr(y), _stream(stream)))


def conv_commit(batch, T, cur, accept, status=None, stream=None):
    _check("conv_commit", load_library().conv_commit(
        batch, T, _ptr(cur), _ptr(accept), _ptr(status), _stream(stream)))


# ------------------------------------------------------------------ convenience owner
_TORCH_DTYPE = {REPLAY_F32: torch.float32, REPLAY_BF16: torch.bfloat16}


class ReplayStore:
    """A store whose workspace is a PyTorch device buffer; keeps A and D alive.

    Methods map one to one onto the C calls. ``region(name)`` returns a typed view of a
    workspace region (for inspection and tests).
    """

    def __init__(self, cfg: ReplayConfig, A: torch.Tensor, D: torch.Tensor, device="cuda",
                 stream=None):
        self.cfg = cfg
        self.layout = replay_layout_of(cfg)
        self.workspace = torch.empty(self.layout.total, dtype=torch.uint8, device=device)
        self.A = A.to(device=device, dtype=torch.float32).contiguous()
        self.D = D.to(device=device, dtype=torch.float32).contiguous()
        self.handle = replay_alloc(cfg, self.workspace, self.layout.total, self.A, self.D, stream)

    def close(self):
        if self.handle:
            replay_free(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def in_dtype(self):
        return _TORCH_DTYPE[self.cfg.in_dtype]

    def step(self, x, B, C, dt, y, stream=None):
        replay_step(self.handle, x, B, C, dt, y, stream)

    def verify(self, T, x, B, C, dt, y, stream=None):
        replay_verify(self.handle, T, x, B, C, dt, y, stream)

    def commit(self, accept, stream=None):
        replay_commit(self.handle, accept, stream)

    def flush(self, stream=None):
        replay_flush(self.handle, stream)

    def reset(self, seq_mask=None, stream=None):
        replay_reset(self.handle, seq_mask, stream)

    def load_state(self, h, stream=None):
        replay_load_state(self.handle, h, stream)

    def export_state(self, h_out, stream=None):
        replay_export_state(self.handle, h_out, stream)

    def status(self, clear=False, stream=None) -> int:
        return replay_status(self.handle, clear, stream)

    def region(self, name: str) -> torch.Tensor:
        c, L = self.cfg, self.layout
        Bz, H, P, N, G, cap = c.batch, c.nheads, c.headdim, c.dstate, c.ngroups, L.cap
        dt = self.in_dtype
        spec = {
            "h0": (torch.float16 if c.checkpoint_format == REPLAY_CKPT_F16_SR else torch.float32,
                   (0,) if c.shared_checkpoint else (Bz, H, P, N)),
            "rc": ({REPLAY_RC_BF16: torch.bfloat16, REPLAY_RC_FP8E4M3: torch.uint8,
                    REPLAY_RC_FP16: torch.float16}.get(c.read_copy, torch.uint8),
                   (Bz, H, P, N // 2) if c.read_copy == REPLAY_RC_NVFP4 else
                   (Bz, H, P, N) if c.read_copy else (0,)),
            "scale": (torch.float32,
                      (Bz, H) if c.read_copy in (REPLAY_RC_FP8E4M3, REPLAY_RC_NVFP4) else (0,)),
            "bscale": (torch.uint8, (Bz, H, P, N // 16) if c.read_copy == REPLAY_RC_NVFP4 else (0,)),
            "xbuf": (dt, (Bz, H, cap, P)), "bbuf": (dt, (Bz, G, cap, N)), "dtbuf": (dt, (Bz, H, cap)),
            "meta": (torch.int32, (Bz, 4)), "arrive": (torch.int32, (Bz,)), "status": (torch.int32, (1,)),
            "plan": (torch.int32, (2, Bz, 4)),
            "coef": (torch.float32, (Bz, H, max(c.max_draft_T + 1, 2), cap + 1)),
        }[name]
        tdt, shape = spec
        nbytes = torch.empty((), dtype=tdt).element_size()
        count = 1
        for s in shape:
            count *= s
        off = getattr(L, name)
        return self.workspace[off: off + count * nbytes].view(tdt).view(shape)
