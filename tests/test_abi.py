"""The C ABI library on the host (no GPU needed): it loads, exports every declared
symbol, computes layouts, and rejects bad arguments before any CUDA call."""
import ctypes

import pytest

from hybrid_model_ssm_mamba_gb300 import replay as R


def test_exports_every_header_symbol(lib):
    names = R.header_functions()
    assert len(names) >= 17
    for n in names:
        assert hasattr(lib, n), n
    assert lib.replay_abi_version() == 4
    assert lib.replay_strerror(-3) == b"capacity exceeded"


def test_layout_of_nemotron_layer():
    cfg = R.ReplayConfig(256, 128, 64, 128, 8, 16, 0, R.REPLAY_BF16, R.REPLAY_RC_NONE)
    L = R.replay_layout_of(cfg)
    assert L.cap == 16
    assert L.h0 == 0 and L.rc == 1 << 30 and L.xbuf == 1 << 30
    assert L.bbuf - L.xbuf == 256 * 128 * 16 * 64 * 2
    assert L.dtbuf - L.bbuf == 256 * 8 * 16 * 128 * 2
    for name in ("h0", "rc", "scale", "xbuf", "bbuf", "dtbuf", "meta", "arrive", "status", "total"):
        assert getattr(L, name) % 256 == 0
    assert R.replay_store_bytes(cfg) == L.total


@pytest.mark.parametrize("T", [0, 1, 4])
def test_layout_step_buffers(T):
    """Consecutive steps alternate between two plans and two coefficient blocks (a step's prep
    may write its own while the previous step's per-head kernel reads the other): the plan
    region holds 2 x batch int4, the coefficient region at least two batch x H x (cap + 1)
    blocks, and a verify's [batch][H][T + 1][cap + 1] when T + 1 > 2."""
    cfg = R.ReplayConfig(64, 16, 64, 128, 2, 8, T, R.REPLAY_BF16, R.REPLAY_RC_BF16)
    L = R.replay_layout_of(cfg)
    block = 64 * 16 * (L.cap + 1) * 4
    assert L.coef - L.plan >= 2 * 64 * 16
    assert L.total - L.coef >= max(T + 1, 2) * block
    assert L.total - L.coef < max(T + 1, 2) * block + 256


def test_layout_ring_capacity_and_read_copies():
    cfg = R.ReplayConfig(512, 8, 64, 128, 1, 16, 4, R.REPLAY_F32, R.REPLAY_RC_FP8E4M3)
    L = R.replay_layout_of(cfg)
    assert L.cap == 16 + 2 * 4 - 1
    assert L.scale - L.rc == 512 * 8 * 64 * 128
    assert L.xbuf - L.scale == 512 * 8 * 4
    for rc in (R.REPLAY_RC_BF16, R.REPLAY_RC_FP16):
        cfg.read_copy = rc
        L = R.replay_layout_of(cfg)
        assert L.scale - L.rc == 512 * 8 * 64 * 128 * 2 and L.xbuf == L.scale


def test_layout_nvfp4_regions():
    cfg = R.ReplayConfig(512, 8, 64, 128, 1, 16, 0, R.REPLAY_F32, R.REPLAY_RC_NVFP4)
    L = R.replay_layout_of(cfg)
    assert L.scale - L.rc == 512 * 8 * 64 * 128 // 2        # two codes per byte
    assert L.bscale - L.scale == 512 * 8 * 4                 # FP32 slab scale
    assert L.xbuf - L.bscale == 512 * 8 * 64 * 128 // 16     # one E4M3 scale per 16 values
    assert R.replay_store_bytes(cfg) == L.total


@pytest.mark.parametrize("rc,dstate", [(R.REPLAY_RC_FP16, 256), (R.REPLAY_RC_NVFP4, 256),
                                       (R.REPLAY_RC_NVFP4, 64)])
def test_copies_without_a_kernel_for_the_dstate(rc, dstate):
    cfg = R.ReplayConfig(4, 8, 64, dstate, 4, 16, 0, R.REPLAY_F32, rc, 1)
    with pytest.raises(R.ReplayError) as e:
        R.replay_layout_of(cfg)
    assert e.value.code == -2


@pytest.mark.parametrize("field,value,code", [
    ("batch", 0, -1), ("nheads", 6, -1), ("ngroups", 0, -1), ("window_L", 0, -1),
    ("max_draft_T", -1, -1), ("in_dtype", 7, -1), ("read_copy", 5, -1), ("headdim", 48, -2),
    ("dstate", 96, -2), ("window_L", 65, -3), ("max_draft_T", 9, -3)])
def test_layout_rejects(field, value, code):
    cfg = R.ReplayConfig(4, 8, 64, 128, 4, 16, 2, R.REPLAY_F32, R.REPLAY_RC_NONE)
    setattr(cfg, field, value)
    with pytest.raises(R.ReplayError) as e:
        R.replay_layout_of(cfg)
    assert e.value.code == code


def test_calls_reject_null_arguments_before_cuda(lib):
    cfg = R.ReplayConfig(4, 8, 64, 128, 4, 16, 2, R.REPLAY_F32, R.REPLAY_RC_NONE)
    out = ctypes.c_void_p()
    assert lib.replay_alloc(ctypes.byref(cfg), None, 1 << 20, None, None, None, ctypes.byref(out)) == -1
    assert lib.replay_alloc(ctypes.byref(cfg), 256, 16, 256, 256, None, ctypes.byref(out)) == -3
    assert lib.replay_alloc(ctypes.byref(cfg), 255, 1 << 40, 256, 256, None, ctypes.byref(out)) == -1
    assert lib.replay_step(None, 256, 256, 256, 256, 256, None) == -1
    assert lib.replay_verify(None, 2, 256, 256, 256, 256, 256, None) == -1
    assert lib.replay_commit(None, 256, None) == -1
    assert lib.replay_flush(None, None) == -1
    assert lib.replay_free(None) == -1
    assert lib.conv_step(ctypes.byref(cfg), None, 0, 256, 256, 256, 256, 256, 256, 256, None) == -1
    assert lib.conv_step(ctypes.byref(cfg), 256, 5, 256, 256, 256, 256, 256, 256, 256, None) == -1
    assert lib.conv_commit(4, 0, 256, 256, None, None) == -1
    bad = R.ReplayConfig(4, 8, 64, 96, 4, 16, 2, R.REPLAY_F32, R.REPLAY_RC_NONE)
    assert lib.conv_step(ctypes.byref(bad), 256, 0, 256, 256, 256, 256, 256, 256, 256, None) == -2


def test_shared_checkpoint_layout_and_rules():
    cfg = R.ReplayConfig(4, 8, 64, 128, 4, 16, 0, R.REPLAY_F32, R.REPLAY_RC_BF16, 1)
    L = R.replay_layout_of(cfg)
    assert L.h0 == 0 and L.rc == 0                 # no FP32 checkpoint region
    assert L.scale - L.rc == 4 * 8 * 64 * 128 * 2
    for rc, shared in ((R.REPLAY_RC_NONE, 1), (R.REPLAY_RC_BF16, 2)):
        cfg = R.ReplayConfig(4, 8, 64, 128, 4, 16, 0, R.REPLAY_F32, rc, shared)
        with pytest.raises(R.ReplayError) as e:
            R.replay_layout_of(cfg)
        assert e.value.code == -1


def test_fp16_checkpoint_layout_and_rules():
    """checkpoint_format = REPLAY_CKPT_F16_SR keeps the recurrence checkpoint in FP16 (half the
    bytes) beside a separate read copy; it needs a bf16, E4M3 or NVFP4 copy, no shared
    checkpoint, and dstate <= 128."""
    cfg = R.ReplayConfig(4, 8, 64, 128, 4, 16, 0, R.REPLAY_F32, R.REPLAY_RC_NVFP4, 0, R.REPLAY_CKPT_F16_SR)
    L = R.replay_layout_of(cfg)
    assert L.h0 == 0 and L.rc == 4 * 8 * 64 * 128 * 2
    for rc, shared, fmt, code in ((R.REPLAY_RC_NONE, 0, 1, -1), (R.REPLAY_RC_FP16, 0, 1, -1),
                                  (R.REPLAY_RC_NVFP4, 1, 1, -1), (R.REPLAY_RC_BF16, 0, 2, -1)):
        bad = R.ReplayConfig(4, 8, 64, 128, 4, 16, 0, R.REPLAY_F32, rc, shared, fmt)
        with pytest.raises(R.ReplayError) as e:
            R.replay_layout_of(bad)
        assert e.value.code == code
    wide = R.ReplayConfig(4, 8, 64, 256, 4, 16, 0, R.REPLAY_F32, R.REPLAY_RC_BF16, 0, R.REPLAY_CKPT_F16_SR)
    with pytest.raises(R.ReplayError) as e:
        R.replay_layout_of(wide)
    assert e.value.code == -2
