"""NVFP4 read copy on the GPU against the oracle's NVFP4 codec and the FP64 recurrence.

Source: "ReplaySSM: Rethinking State Storage for Faster Hybrid-Model Decoding", sections
"Benefit 3" (a flush casts the new FP32 checkpoint independently into the low-precision
copy; non-flush steps read only the copy) and "State quantization" (NVFP4 reads).

Checked, bit for bit: the codes, block scales and slab scale a checkpoint write produces,
against the oracle's encoder applied to the same FP32 state (codes decided in FP32 on both
sides; +0 and -0 codes are the same value). Within 1e-4 (FP32 arithmetic): non-flush outputs
against the unrolled window evaluated in FP64 from the oracle's dequantized copy, and flush
outputs and checkpoints against the exact recurrence. Three kernels read the copy: the fused
small-call kernel, the NVFP4 kernel (one warp per head, h0 . C on the tensor cores), and the
one-head-per-CTA kernel.
"""
import numpy as np
import pytest
import torch

import synthgen as sg
from gpu_util import dev, rel_vec_err
from hybrid_model_ssm_mamba_gb300 import replay as R
from oracle import formats as F
from oracle.mamba2 import Mamba2Decoder, window_output

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _store(shape, seed, L, shared=0):
    A, D = sg.head_params(shape.nheads, seed)
    dt = R.REPLAY_F32 if shape.dtype == "f32" else R.REPLAY_BF16
    cfg = R.ReplayConfig(shape.batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, L, 0, dt,
                         R.REPLAY_RC_NVFP4, shared)
    return R.ReplayStore(cfg, torch.from_numpy(A), torch.from_numpy(D)), A.astype(float), D.astype(float)


def _oracle_copy(h32):
    """The oracle's NVFP4 encoding of FP32 states [b, H, P, N]: packed codes, block-scale
    codes, slab scales, and the values read back."""
    b, H, P, N = h32.shape
    q = np.empty((b, H, P, N), np.uint8)
    sb = np.empty((b, H, P, N // 16), np.uint8)
    sg_ = np.empty((b, H), np.float32)
    back = np.empty((b, H, P, N))
    for i in range(b):
        for h in range(H):
            q[i, h], sb[i, h], sg_[i, h] = F.nvfp4_slab_quantize(h32[i, h])
            back[i, h] = F.nvfp4_slab_dequantize(q[i, h], sb[i, h], sg_[i, h])
    return q, sb, sg_, back


def device_codes(rc):
    """E2M1 codes [..., P, 128] from the library's NVFP4 row layout [..., P, 64] bytes, as
    the header defines it: quarter u of block b is the 2-byte unit at byte 16u + 2b; byte 0
    holds columns 16b+4u (slot A) and 16b+4u+2 (slot B), byte 1 columns 16b+4u+1 (A) and
    16b+4u+3 (B); slot A = sign bit 7, magnitude bits 3..1; slot B = sign bit 0, magnitude
    bits 6..4."""
    rc = np.asarray(rc, dtype=np.uint8)
    out = np.empty(rc.shape[:-1] + (128,), dtype=np.uint8)
    slot_a = lambda v: ((v >> 4) & 8) | ((v >> 1) & 7)
    slot_b = lambda v: ((v & 1) << 3) | ((v >> 4) & 7)
    for u in range(4):
        for b in range(8):
            b0, b1 = rc[..., 16 * u + 2 * b], rc[..., 16 * u + 2 * b + 1]
            c = 16 * b + 4 * u
            out[..., c], out[..., c + 2] = slot_a(b0), slot_b(b0)
            out[..., c + 1], out[..., c + 3] = slot_a(b1), slot_b(b1)
    return out


def _assert_copy_is_encoding_of(st, h32, seqs):
    q, sb, sgl, _ = _oracle_copy(h32)
    assert np.array_equal(st.region("scale").cpu().numpy()[seqs], sgl)
    assert np.array_equal(st.region("bscale").cpu().numpy()[seqs], sb)
    got = device_codes(st.region("rc").cpu().numpy()[seqs])
    same = (got == q) | (((got & 7) == 0) & ((q & 7) == 0))           # +-0 both zero
    assert same.all(), np.argwhere(~same)[:4]


@pytest.mark.parametrize("shared", [0, 1])
def test_nvfp4_codes_match_format_definition(shared):
    shape = sg.LayerShape(3, 4, 64, 128, 1, "f32")
    st, _, _ = _store(shape, 9, 4, shared)
    h = sg.initial_state(shape, 9)
    h[0, 1] = 0.0                                   # an all-zero slab: s_g = 1, zero codes
    h[1, 2, 0, :4] = [1e-12, -3e-9, 500.0, -1e30]   # a huge value: every other block scale tiny
    h[2, 3, 5, 16:32] = 0.0                         # an all-zero block: s_b = 0
    # Exact E2M1 ties: slab (2, 0) has absmax 5.25, so s_g = 2**-9; a block with absmax 3
    # gets s_b = 256 and e = 0.5, and holds every midpoint between E2M1 values times e.
    h[2, 0] = np.clip(h[2, 0], -1.0, 1.0)
    h[2, 0, 0, 0] = 5.25
    h[2, 0, 7, :16] = 0.5 * np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 2)
    st.load_state(torch.from_numpy(h).cuda())
    _assert_copy_is_encoding_of(st, h, np.arange(3))
    assert st.region("scale").cpu().numpy()[2, 0] == 2.0 ** -9
    assert F.e2m1_decode(device_codes(st.region("rc").cpu().numpy())[2, 0, 7, :8]).tolist() == \
        [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0]
    if shared:   # the copy is the state: export reads it back
        out = torch.empty(3, 4, 64, 128, device="cuda")
        st.export_state(out)
        assert np.array_equal(out.cpu().numpy(), _oracle_copy(h)[3].astype(np.float32))


def test_nvfp4_codes_at_rounding_boundaries():
    """Every block holds its maximum and fifteen elements placed within a few ulps of E2M1
    midpoints (and of the 0.25 boundary) times the block's scale unit e, both signs; block
    maxima vary so that e is rarely a power of two. Codes, block scales and slab scales equal
    the encoder's, bit for bit."""
    shape = sg.LayerShape(1, 2, 64, 128, 1, "f32")
    st, _, _ = _store(shape, 9, 4)
    rng = np.random.default_rng(13)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    h = np.empty((1, 2, 64, 128), np.float32)
    for hh, amax in enumerate((2688.0 * 0.731, 2688.0 * 3.3e-3)):
        sg_ = np.float32(np.float32(amax) / np.float32(2688.0))
        blocks = h[0, hh].reshape(-1, 16)
        for j, blk in enumerate(blocks):
            bm = np.float32(amax if j == 0 else amax * rng.uniform(0.05, 1.0))
            sb = F.e4m3_encode(np.float32(bm / np.float32(6.0 * sg_)))
            e = np.float32(F.e4m3_decode(sb)) * sg_
            blk[0] = bm
            for i in range(1, 16):
                m, k, sgn = mids[(i + j) % 7], (i * 7 + j) % 11 - 5, 1 if (i + j) % 2 else -1
                blk[i] = sgn * _near(np.float32(m) * np.float32(e), k)
            blk[1:] = np.clip(blk[1:], -bm, bm)
    st.load_state(torch.from_numpy(h).cuda())
    _assert_copy_is_encoding_of(st, h, np.arange(1))


def _near(v, k):
    """FP32 values k ulps from v (k < 0: toward zero)."""
    v = np.float32(v)
    for _ in range(abs(k)):
        v = np.nextafter(v, np.float32(np.inf) if (k > 0) == (v > 0) else np.float32(0))
    return v


# (batch, heads, groups): the fused kernel (batch * heads <= 1024); the NVFP4 tensor-core kernel
# (heads per group a multiple of 8); the one-head-per-CTA kernel (6 heads per group). A flush the
# host sees coming takes the one-head-per-CTA kernel; after a masked reset (here of no
# sequence) the host no longer knows the ring counts and every step takes the read kernel,
# flushes included.
@pytest.mark.parametrize("batch,heads,groups,dtype,known", [
    (4, 8, 1, "f32", True), (72, 128, 8, "bf16", True), (72, 128, 8, "bf16", False),
    (96, 12, 2, "f32", True), (96, 12, 2, "f32", False), (17, 64, 8, "bf16", True), (23, 64, 4, "f32", True)])
def test_nvfp4_reads_and_flushes_follow_the_oracle(batch, heads, groups, dtype, known):
    shape = sg.LayerShape(batch, heads, 64, 128, groups, dtype)
    L, seed = 8, 23
    st, A, D = _store(shape, seed, L)
    sel = np.array([0, batch // 2, batch - 1])
    h0 = sg.initial_state(shape, seed)
    st.load_state(torch.from_numpy(h0).cuda())
    if not known:
        st.reset(torch.zeros(batch, dtype=torch.int32, device="cuda"))
    orc = Mamba2Decoder(A, D, groups, h0[sel].astype(np.float64))
    ckpt = h0[sel]                                   # FP32 checkpoint the copy was cast from
    y = torch.empty(batch, heads, 64, device="cuda")
    d = sg.token_inputs(shape, seed, np.arange(3 * L))
    rec = {k: [] for k in ("x", "B", "dt")}
    worst_read = worst_flush = 0.0
    for t in range(3 * L):
        devs = [dev(_tok(d[k], t), dtype) for k in ("x", "B", "C", "dt")]
        st.step(*devs, y)
        f64 = [d[k].f64[sel, t] for k in ("x", "B", "C", "dt")]
        for k, v in zip(("x", "B", "dt"), (f64[0], f64[1], f64[3])):
            rec[k].append(v)
        yref = orc.step(*f64)
        yg = y[sel].cpu().numpy()
        if (t + 1) % L:      # non-flush: the window from the dequantized copy
            hread = _oracle_copy(ckpt)[3]
            ywin = window_output(hread, np.stack(rec["x"], 1), np.stack(rec["B"], 1), np.stack(rec["dt"], 1),
                                 f64[2], A, D)
            worst_read = max(worst_read, rel_vec_err(yg, ywin, 2).max())
        else:                # flush: the exact recurrence, and the new copy from the new FP32 state
            worst_flush = max(worst_flush, rel_vec_err(yg, yref, 2).max())
            out = torch.empty(batch, heads, 64, 128, device="cuda")
            st.export_state(out)
            ckpt = out.cpu().numpy()[sel]
            assert rel_vec_err(ckpt, orc.h, 2).max() <= TOL
            _assert_copy_is_encoding_of(st, ckpt, sel)
            rec = {k: [] for k in ("x", "B", "dt")}
    assert worst_read <= TOL and worst_flush <= TOL, (worst_read, worst_flush)
    assert st.status() == 0


def test_nvfp4_read_error_is_bounded():
    """Against the exact recurrence the copy's read error is reported, not bounded by the
    pages; here it stays an NVFP4-sized error and does not grow across windows."""
    shape = sg.LayerShape(72, 128, 64, 128, 8, "bf16")
    L, seed = 16, 29
    st, A, D = _store(shape, seed, L)
    sel = np.array([5, 40])
    orc = Mamba2Decoder(A, D, 8, np.zeros((2, 128, 64, 128)))
    y = torch.empty(72, 128, 64, device="cuda")
    d = sg.token_inputs(shape, seed, np.arange(4 * L))
    errs = []
    for t in range(4 * L):
        devs = [dev(_tok(d[k], t), "bf16") for k in ("x", "B", "C", "dt")]
        st.step(*devs, y)
        yref = orc.step(*(d[k].f64[sel, t] for k in ("x", "B", "C", "dt")))
        errs.append(rel_vec_err(y[sel].cpu().numpy(), yref, 2).mean())
    errs = np.array(errs).reshape(4, L)
    assert errs.max() <= 0.2
    assert errs[-1].mean() <= 2.0 * errs[1].mean() + 1e-6
    assert st.status() == 0


class _Tok:
    def __init__(self, store, f64):
        self.store, self.f64 = store, f64


def _tok(drawn, t):
    return _Tok(np.ascontiguousarray(drawn.store[:, t]), drawn.f64[:, t])
