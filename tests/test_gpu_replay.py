"""GPU parity of the replay path against the FP64 oracle, through the C ABI.

Bar (FP32 path): every output vector and every checkpoint slab within 1e-4 relative
(inf-norm per vector, see gpu_util); bf16 read copy within 1e-2; integer metadata exact.
"""
import numpy as np
import pytest
import torch

import synthgen as sg
from gpu_util import DTYPE, draft_device, make_store, rel_vec_err, step_inputs
from hybrid_model_ssm_mamba_gb300 import replay as R
from oracle import formats as F
from oracle.mamba2 import Mamba2Decoder, window_output
from test_gpu_nvfp4 import device_codes

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def run_decode(shape, steps, L, seed=0, read_copy=R.REPLAY_RC_NONE, seqs=None, check_ckpt=True,
               on_step=None, T=0):
    """Decode `steps` tokens on the GPU and in the oracle (sequences `seqs`); returns the
    worst output error, the worst post-flush checkpoint error and the store."""
    st, A, D = make_store(shape, seed, L=L, T=T, read_copy=read_copy)
    sel = np.arange(shape.batch) if seqs is None else np.asarray(seqs)
    H, P, N = shape.nheads, shape.headdim, shape.dstate
    orc = Mamba2Decoder(A, D, shape.ngroups, np.zeros((len(sel), H, P, N)))
    y = torch.empty(shape.batch, H, P, device="cuda")
    worst_y = worst_h = 0.0
    for t in range(steps):
        devs, f64 = step_inputs(shape, seed, t, sel)
        st.step(*devs, y)
        yref = orc.step(*f64)
        worst_y = max(worst_y, rel_vec_err(y[sel].cpu().numpy(), yref, 2).max())
        if check_ckpt and (t + 1) % L == 0:
            h0 = st.region("h0")[sel].cpu().numpy()
            worst_h = max(worst_h, rel_vec_err(h0, orc.h, 2).max())
        if on_step is not None:
            on_step(t, st, orc)
    torch.cuda.synchronize()
    assert st.status() == 0
    return worst_y, worst_h, st, orc


def test_tiny_layer_all_steps():
    """Tiny Mamba-2 layer: batch 1, 8 heads, P 64, N 128, G 1, FP32, L 16, 64 steps."""
    shape = sg.LayerShape(1, 8, 64, 128, 1, "f32")
    wy, wh, st, orc = run_decode(shape, 64, 16)
    assert wy <= TOL and wh <= TOL, (wy, wh)
    meta = st.region("meta").cpu().numpy()
    assert meta[0, 1] == 0 and meta[0, 2] == 0           # 64 = 4 windows: ring empty
    assert meta[0, 3] == 5                               # the load was write 0, then 4 flushes


@pytest.mark.parametrize("N,dtype,G,L,steps", [
    (128, "bf16", 2, 5, 13), (64, "f32", 3, 7, 17), (256, "bf16", 1, 4, 9), (128, "f32", 6, 1, 5),
    (128, "f32", 2, 40, 45)])
def test_ragged_shapes(N, dtype, G, L, steps):
    """Odd batch and head counts, several group sizes, windows that do not divide the run."""
    shape = sg.LayerShape(3, 6, 64, N, G, dtype)
    wy, wh, st, orc = run_decode(shape, steps, L, seed=3)
    assert wy <= TOL and wh <= TOL, (wy, wh)
    meta = st.region("meta").cpu().numpy()
    assert np.all(meta[:, 1] == steps % L)
    assert np.all(meta[:, 0] == (steps - steps % L) % L)
    h = torch.empty(3, 6, 64, N, device="cuda")
    st.export_state(h)
    assert rel_vec_err(h.cpu().numpy(), orc.h, 2).max() <= TOL


def test_export_does_not_mutate_and_load_roundtrips():
    shape = sg.LayerShape(2, 4, 64, 128, 2, "f32")
    st, A, D = make_store(shape, 1, L=8)
    h0 = torch.from_numpy(sg.initial_state(shape, 1)).cuda()
    st.load_state(h0)
    out = torch.empty_like(h0)
    st.export_state(out)
    assert torch.equal(out, h0)
    orc = Mamba2Decoder(A, D, 2, h0.cpu().numpy().astype(np.float64))
    y = torch.empty(2, 4, 64, device="cuda")
    for t in range(11):
        devs, f64 = step_inputs(shape, 1, t)
        st.step(*devs, y)
        assert rel_vec_err(y.cpu().numpy(), orc.step(*f64), 2).max() <= TOL
    meta_before = st.region("meta").clone()
    h0_before = st.region("h0").clone()
    st.export_state(out)
    st.export_state(out)
    assert torch.equal(st.region("meta"), meta_before) and torch.equal(st.region("h0"), h0_before)
    assert rel_vec_err(out.cpu().numpy(), orc.h, 2).max() <= TOL


def test_forced_flush_and_staggered_phases():
    """replay_flush mid-window, and per-sequence resets that leave sequences in different
    phases within one launch."""
    shape = sg.LayerShape(4, 4, 64, 128, 1, "bf16")
    st, A, D = make_store(shape, 2, L=6)
    orc = Mamba2Decoder(A, D, 1, np.zeros((4, 4, 64, 128)))
    y = torch.empty(4, 4, 64, device="cuda")
    for t in range(23):
        devs, f64 = step_inputs(shape, 2, t)
        if t == 4:
            st.flush()
            assert st.region("meta").cpu().numpy()[:, 1].tolist() == [0, 0, 0, 0]
        if t in (7, 15):
            mask = torch.tensor([0, 1, 0, 1] if t == 7 else [1, 0, 0, 0], dtype=torch.int32, device="cuda")
            st.reset(mask)
            orc.h[mask.cpu().numpy().astype(bool)] = 0.0
        st.step(*devs, y)
        assert rel_vec_err(y.cpu().numpy(), orc.step(*f64), 2).max() <= TOL, t
    n = st.region("meta").cpu().numpy()[:, 1]
    assert len(set(n.tolist())) > 1          # the sequences really are out of phase
    assert st.status() == 0


@pytest.mark.parametrize("L", [1, 4, 8, 16, 32])
def test_window_length_invariance(L):
    """Outputs do not depend on the window; L = 1 is the conventional step."""
    shape = sg.LayerShape(2, 8, 64, 128, 2, "f32")
    wy, wh, _, _ = run_decode(shape, 40, L, seed=5)
    assert wy <= TOL and wh <= TOL, (L, wy, wh)


@pytest.mark.parametrize("batch,heads,groups,dtype,read_copy", [
    (2, 8, 2, "f32", R.REPLAY_RC_NONE), (72, 128, 8, "bf16", R.REPLAY_RC_NONE),
    (72, 128, 8, "bf16", R.REPLAY_RC_BF16), (72, 128, 8, "f32", R.REPLAY_RC_FP8E4M3)])
def test_longest_window(batch, heads, groups, dtype, read_copy):
    """L = 64, the most records a ring holds without verify: non-flush steps with more than 32
    buffered records (lanes s and s + 32 both carry records), one flush of 64 records; the
    read-copy kernels with their largest record staging (the E4M3 tensor-core read with FP32
    inputs stages 64 records of 4 heads)."""
    shape = sg.LayerShape(batch, heads, 64, 128, groups, dtype)
    wy, wh, _, _ = run_decode(shape, 72, 64, seed=37, read_copy=read_copy, seqs=[0, batch - 1])
    bound = {R.REPLAY_RC_NONE: TOL, R.REPLAY_RC_BF16: 1e-2}.get(read_copy, 0.25)  # E4M3: vs the FP32 state
    assert wy <= bound and wh <= TOL, (wy, wh)


@pytest.mark.parametrize("N,dtype,L,T", [
    (128, "f32", 16, 0), (128, "bf16", 9, 2), (64, "f32", 3, 0), (64, "bf16", 24, 0),
    (256, "f32", 13, 0), (256, "bf16", 1, 0)])
def test_known_flush_on_the_large_call_path(N, dtype, L, T):
    """A flush the host sees coming, on a call of more than 1024 slabs (the prep kernel and
    the flush instantiation of the bulk-copy read kernel: records staged while the slab
    lands, fold from shared memory):
    every dstate, both input types, folds of 1 to 24 records, and a ring sized for verify
    (T = 2). Outputs and checkpoints against the FP64 oracle at the FP32 bar."""
    shape = sg.LayerShape(40, 32, 64, N, 4, dtype)
    wy, wh, st, _ = run_decode(shape, 2 * L + 3, L, seed=41, seqs=[0, 17, 39], T=T)
    assert st.layout.cap == (L + 2 * T - 1 if T else L)
    assert wy <= TOL and wh <= TOL, (wy, wh)


@pytest.mark.parametrize("rc,bound", [(R.REPLAY_RC_NONE, TOL), (R.REPLAY_RC_BF16, 1e-2),
                                      (R.REPLAY_RC_FP8E4M3, 0.25), (R.REPLAY_RC_NVFP4, 0.25)])
def test_wrong_phase_hint_still_follows_the_oracle(rc, bound):
    """The host's count of buffered records only picks kernels; every kernel follows the
    plan the device reads from the ring metadata. Here the device state is rewound behind
    the host's back (regions restored after two extra steps), so the host expects a flush
    where the ring holds one record (the flush kernel meets a non-flush plan), and later a
    non-flush step where the ring is full (the bulk-copy read kernels, FP32 or read copy, and
    the NVFP4 kernel meet a flush plan). Non-flush outputs read the copy (its bound); flush
    outputs and checkpoints follow the oracle at 1e-4."""
    shape = sg.LayerShape(40, 32, 64, 128, 4, "bf16")
    L, seed, sel = 4, 43, np.array([0, 21, 39])
    st, A, D = make_store(shape, seed, L=L, read_copy=rc)
    orc = Mamba2Decoder(A, D, 4, np.zeros((3, 32, 64, 128)))
    y = torch.empty(40, 32, 64, device="cuda")

    def step(t):
        devs, f64 = step_inputs(shape, seed, t, sel)
        st.step(*devs, y)
        err = rel_vec_err(y[sel].cpu().numpy(), orc.step(*f64), 2).max()
        return err <= (TOL if t in (3, 7) else bound)

    assert step(0)
    names = ("h0", "meta", "xbuf", "bbuf", "dtbuf") + (("rc",) if rc else ()) + \
        (("scale",) if rc in (R.REPLAY_RC_FP8E4M3, R.REPLAY_RC_NVFP4) else ()) + \
        (("bscale",) if rc == R.REPLAY_RC_NVFP4 else ())
    saved = {k: st.region(k).clone() for k in names}
    for t in (100, 101):                             # steps the oracle does not see
        devs, _ = step_inputs(shape, seed, t)
        st.step(*devs, y)
    for k in names:
        st.region(k).copy_(saved[k])
    for t in range(1, 8):                            # the device flushes after tokens 3 and 7
        assert step(t), t
        if t in (3, 7):
            h0 = st.region("h0")[sel].cpu().numpy()
            assert rel_vec_err(h0, orc.h, 2).max() <= TOL, t
            assert np.all(st.region("meta").cpu().numpy()[:, 1] == 0)
    assert st.status() == 0


def test_verify_fullest_ring():
    """L = 49 and T = 8 give a ring of 64 records; commits of all drafts push the committed
    count to L - 1 + T = 56 before a verify pre-folds, so record lanes past 32 are used."""
    shape = sg.LayerShape(4, 8, 64, 128, 2, "f32")
    T, L = 8, 49
    st, A, D = make_store(shape, 39, L=L, T=T)
    assert st.layout.cap == 64
    orc = Mamba2Decoder(A, D, 2, np.zeros((4, 8, 64, 128)))
    y = torch.empty(4, T, 8, 64, device="cuda")
    worst = 0.0
    for call in range(10):
        devs, f64 = draft_device(shape, 39, call, T)
        st.verify(T, *devs, y)
        worst = max(worst, rel_vec_err(y.cpu().numpy(), orc.verify(*f64), 3).max())
        acc = np.full(4, T, dtype=np.int32)
        acc[1] = call % (T + 1)
        st.commit(torch.from_numpy(acc).cuda())
        orc.commit(acc, f64[0], f64[1], f64[3])
    assert worst <= TOL, worst
    h = torch.empty(4, 8, 64, 128, device="cuda")
    st.export_state(h)
    assert rel_vec_err(h.cpu().numpy(), orc.h, 2).max() <= TOL
    assert st.status() == 0


def test_replay_equals_conventional_gpu():
    """GPU replay == GPU load-update-store on the same inputs (bf16 inputs, FP32 state)."""
    shape = sg.LayerShape(4, 16, 64, 128, 4, "bf16")
    st, A, D = make_store(shape, 6, L=16)
    cfg = st.cfg
    state = torch.zeros(4, 16, 64, 128, device="cuda")
    y1 = torch.empty(4, 16, 64, device="cuda")
    y2 = torch.empty_like(y1)
    for t in range(35):
        devs, _ = step_inputs(shape, 6, t)
        st.step(*devs, y1)
        R.conv_step(cfg, state, R.REPLAY_F32, st.A, st.D, *devs, y2)
        assert rel_vec_err(y1.cpu().numpy(), y2.cpu().numpy(), 2).max() <= TOL, t
    h = torch.empty_like(state)
    st.export_state(h)
    assert rel_vec_err(h.cpu().numpy(), state.cpu().numpy(), 2).max() <= TOL


def test_nemotron_layer_sampled_sequences():
    """Nemotron-shaped layer at full size (batch 256, 128 heads, G 8, bf16 inputs, L 16,
    256 steps = 16 flushes), in the launch configuration the benchmark times; the oracle
    follows four seeded sequences (all heads, every step and every checkpoint)."""
    shape = sg.LayerShape(256, 128, 64, 128, 8, "bf16")
    seqs = np.sort(np.random.default_rng(0).choice(256, 4, replace=False))
    wy, wh, st, _ = run_decode(shape, 256, 16, seed=0, seqs=seqs)
    assert wy <= TOL and wh <= TOL, (wy, wh)
    meta = st.region("meta").cpu().numpy()
    assert np.all(meta[:, 1] == 0) and np.all(meta[:, 0] == 0)


def test_read_copy_bf16_bound():
    """bf16 read copy: non-flush outputs within 1e-2 of the FP64 oracle."""
    shape = sg.LayerShape(8, 8, 64, 128, 1, "f32")
    wy, wh, _, _ = run_decode(shape, 48, 16, seed=7, read_copy=R.REPLAY_RC_BF16)
    assert wy <= 1e-2 and wh <= TOL, (wy, wh)


def test_read_copy_fp8_drift_is_bounded():
    """E4M3 read copy: drift is reported, not bounded by the pages; check it stays an
    E4M3-sized read error (no growth) and the FP32 checkpoints stay exact."""
    shape = sg.LayerShape(8, 8, 64, 128, 1, "f32")
    wy, wh, _, _ = run_decode(shape, 64, 16, seed=8, read_copy=R.REPLAY_RC_FP8E4M3)
    assert wh <= TOL and wy <= 0.25, (wy, wh)


@pytest.mark.parametrize("rc,shared", [(R.REPLAY_RC_BF16, 0), (R.REPLAY_RC_FP8E4M3, 0),
                                       (R.REPLAY_RC_FP16, 0), (R.REPLAY_RC_FP16, 1)])
def test_read_copy_codes_match_format_definitions(rc, shared):
    """The copy written by a checkpoint write equals the format encoders applied to the
    same FP32 state, bit for bit (codes decided in FP32 on both sides). A shared FP16
    checkpoint is rounded stochastically with the draws of write number 0."""
    shape = sg.LayerShape(3, 4, 64, 128, 1, "f32")
    A, D = sg.head_params(4, 9)
    cfg = R.ReplayConfig(3, 4, 64, 128, 1, 4, 0, R.REPLAY_F32, rc, shared)
    st = R.ReplayStore(cfg, torch.from_numpy(A), torch.from_numpy(D))
    h = sg.initial_state(shape, 9)
    h[0, 1] = 0.0                                  # an all-zero slab: scale 1
    h[1, 2, 0, :4] = [1e-12, -3e-9, 500.0, -1e30]  # tiny, subnormal-range and huge values
    h[2, 3, 5, :3] = [7e4, -65504.0, 3e-8]         # FP16: past the largest finite, at it, subnormal
    st.load_state(torch.from_numpy(h).cuda())
    got = st.region("rc").cpu()
    if rc == R.REPLAY_RC_BF16:
        assert np.array_equal(got.view(torch.int16).numpy().view(np.uint16), F.bf16_encode(h))
    elif rc == R.REPLAY_RC_FP16 and not shared:
        assert np.array_equal(got.view(torch.int16).numpy().view(np.uint16), F.fp16_encode(h))
    elif rc == R.REPLAY_RC_FP16:
        want = F.fp16_sr_round_state(h, 0, np.arange(3), 3 * 4)
        assert np.array_equal(got.double().numpy(), want)
        assert np.abs(want[2, 3, 5, 0]) == 65504.0          # saturated, not infinite
        assert st.region("meta").cpu().numpy()[:, 3].tolist() == [1, 1, 1]
    else:
        scale = st.region("scale").cpu().numpy()
        for b in range(3):
            for hh in range(4):
                q, s = F.fp8_slab_quantize(h[b, hh])
                assert np.float32(scale[b, hh]) == s
                g = got.numpy()[b, hh]
                same = (g == q) | ((g & 0x7F) == 0) & ((q & 0x7F) == 0)   # +-0 both zero
                assert same.all(), (b, hh, np.argwhere(~same)[:3])


def _near(v, k):
    """FP32 values k ulps from v (k < 0: toward zero)."""
    v = np.float32(v)
    for _ in range(abs(k)):
        v = np.nextafter(v, np.float32(np.inf) if (k > 0) == (v > 0) else np.float32(0))
    return v


def test_e4m3_codes_at_rounding_boundaries():
    """Elements placed within a few ulps of every E4M3 midpoint (times a slab scale that is
    not a power of two, so the quotient is rounded), on both sides and with both signs: the
    codes still equal the encoder applied to the IEEE FP32 quotient, bit for bit."""
    shape = sg.LayerShape(1, 2, 64, 128, 1, "f32")
    A, D = sg.head_params(2, 9)
    cfg = R.ReplayConfig(1, 2, 64, 128, 1, 4, 0, R.REPLAY_F32, R.REPLAY_RC_FP8E4M3)
    st = R.ReplayStore(cfg, torch.from_numpy(A), torch.from_numpy(D))
    rng = np.random.default_rng(12)
    h = (rng.standard_normal((1, 2, 64, 128)) * 0.01).astype(np.float32)
    grid = F.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (grid[:-1] + grid[1:]) / 2                            # every boundary, subnormals included
    for hh, amax in enumerate((448.0 * 1.3711, 448.0 * 0.0173)):
        flat = h[0, hh].reshape(-1)
        flat[0] = amax
        scale = np.float32(np.float32(amax) / np.float32(448.0))
        vals = [_near(np.float32(m) * scale, k) * sgn for m in mids for k in range(-5, 6) for sgn in (1, -1)]
        flat[1:1 + len(vals)] = vals
    st.load_state(torch.from_numpy(h).cuda())
    got = st.region("rc").cpu().numpy()
    for hh in range(2):
        q, s = F.fp8_slab_quantize(h[0, hh])
        assert np.float32(st.region("scale").cpu().numpy()[0, hh]) == s
        same = (got[0, hh] == q) | ((got[0, hh] & 0x7F) == 0) & ((q & 0x7F) == 0)
        assert same.all(), (hh, np.argwhere(~same)[:3])


def test_verify_commit_matches_oracle():
    """Speculative verify + commit with accept ~ U{0..T}, interleaved with decode steps:
    every verify output and the final state match an oracle that decodes only the
    accepted prefixes."""
    shape = sg.LayerShape(8, 8, 64, 128, 2, "f32")
    T, L = 4, 8
    st, A, D = make_store(shape, 11, L=L, T=T)
    orc = Mamba2Decoder(A, D, 2, np.zeros((8, 8, 64, 128)))
    y = torch.empty(8, T, 8, 64, device="cuda")
    y1 = torch.empty(8, 8, 64, device="cuda")
    worst = 0.0
    for call in range(24):
        if call % 5 == 4:
            devs, f64 = step_inputs(shape, 11, 1000 + call)
            st.step(*devs, y1)
            worst = max(worst, rel_vec_err(y1.cpu().numpy(), orc.step(*f64), 2).max())
        devs, f64 = draft_device(shape, 11, call, T)
        st.verify(T, *devs, y)
        worst = max(worst, rel_vec_err(y.cpu().numpy(), orc.verify(*f64), 3).max())
        acc = sg.accept_lengths(8, T, 11, call)
        if call == 3:
            acc[:] = 0
        if call == 6:
            acc[:] = T
        st.commit(torch.from_numpy(acc).cuda())
        orc.commit(acc, f64[0], f64[1], f64[3])
        meta = st.region("meta").cpu().numpy()
        assert np.all(meta[:, 1] <= L - 1 + T) and np.all(meta[:, 2] == 0)
    assert worst <= TOL, worst
    h = torch.empty(8, 8, 64, 128, device="cuda")
    st.export_state(h)
    assert rel_vec_err(h.cpu().numpy(), orc.h, 2).max() <= TOL
    assert st.status() == 0


@pytest.mark.parametrize("rc", [R.REPLAY_RC_NONE, R.REPLAY_RC_BF16])
def test_verify_workload_shape(rc):
    """The speculative workload's shape (batch 512, 8 heads, T 4, ring of 23), 20 verify
    calls; the oracle follows 6 seeded sequences."""
    shape = sg.LayerShape(512, 8, 64, 128, 1, "f32")
    T, L = 4, 16
    st, A, D = make_store(shape, 12, L=L, T=T, read_copy=rc)
    assert st.layout.cap == 23
    sel = np.array([0, 77, 200, 311, 480, 511])
    orc = Mamba2Decoder(A, D, 1, np.zeros((6, 8, 64, 128)))
    y = torch.empty(512, T, 8, 64, device="cuda")
    worst = 0.0
    for call in range(20):
        devs, f64 = draft_device(shape, 12, call, T)
        st.verify(T, *devs, y)
        f64s = [a[sel] for a in f64]
        worst = max(worst, rel_vec_err(y[sel].cpu().numpy(), orc.verify(*f64s), 3).max())
        acc = sg.accept_lengths(512, T, 12, call)
        st.commit(torch.from_numpy(acc).cuda())
        orc.commit(acc[sel], f64s[0], f64s[1], f64s[3])
    bound = TOL if rc == R.REPLAY_RC_NONE else 1e-2
    assert worst <= bound, worst
    assert st.status() == 0


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6, 7, 8])
def test_verify_draft_counts_bf16(T):
    """Every draft count: the packed-FMA kernel (T not a multiple of 4) and the tensor-core
    kernel (T = 4, 8), bf16 inputs, 4 groups; commits leave up to L - 1 + T records so that
    verifies also pre-fold. Every output and the final state against the oracle."""
    shape = sg.LayerShape(6, 16, 64, 128, 4, "bf16")
    L = 8
    st, A, D = make_store(shape, 13, L=L, T=T)
    orc = Mamba2Decoder(A, D, 4, np.zeros((6, 16, 64, 128)))
    y = torch.empty(6, T, 16, 64, device="cuda")
    worst = 0.0
    for call in range(12):
        devs, f64 = draft_device(shape, 13, call, T)
        st.verify(T, *devs, y)
        worst = max(worst, rel_vec_err(y.cpu().numpy(), orc.verify(*f64), 3).max())
        acc = sg.accept_lengths(6, T, 13, call)
        if call % 4 == 1:
            acc[:] = T
        st.commit(torch.from_numpy(acc).cuda())
        orc.commit(acc, f64[0], f64[1], f64[3])
    assert worst <= TOL, worst
    h = torch.empty(6, 16, 64, 128, device="cuda")
    st.export_state(h)
    assert rel_vec_err(h.cpu().numpy(), orc.h, 2).max() <= TOL
    assert st.status() == 0


@pytest.mark.parametrize("rc,shared", [(R.REPLAY_RC_BF16, 0), (R.REPLAY_RC_FP16, 0), (R.REPLAY_RC_FP8E4M3, 0),
                                       (R.REPLAY_RC_NVFP4, 0), (R.REPLAY_RC_BF16, 1), (R.REPLAY_RC_FP8E4M3, 1)])
def test_verify_reads_the_decoded_copy(rc, shared):
    """Verify with a read copy (or a shared low-precision checkpoint) evaluates every draft
    from the copy: six verify + commit calls (no pre-fold: L 32, T 4) against the oracle
    started from the copy's decoded values of the loaded state, within 1e-4 (40 sequences x
    32 heads, 4 groups, bf16 inputs)."""
    shape = sg.LayerShape(40, 32, 64, 128, 4, "bf16")
    T, L, seed = 4, 32, 19
    A, D = sg.head_params(32, seed)
    cfg = R.ReplayConfig(40, 32, 64, 128, 4, L, T, DTYPE["bf16"], rc, shared)
    st = R.ReplayStore(cfg, torch.from_numpy(A), torch.from_numpy(D))
    A, D = A.astype(np.float64), D.astype(np.float64)
    sel = np.array([0, 21, 39])
    h0 = sg.initial_state(shape, seed)
    st.load_state(torch.from_numpy(h0).cuda())
    hdec = F.nvfp4_round_state(h0[sel]) if rc == R.REPLAY_RC_NVFP4 else _decoded_copy(st, rc, h0[sel])
    orc = Mamba2Decoder(A, D, 4, hdec)
    y = torch.empty(40, T, 32, 64, device="cuda")
    worst = 0.0
    for call in range(6):
        devs, f64 = draft_device(shape, seed, call, T)
        st.verify(T, *devs, y)
        f64s = [a[sel] for a in f64]
        worst = max(worst, rel_vec_err(y[sel].cpu().numpy(), orc.verify(*f64s), 3).max())
        acc = sg.accept_lengths(40, T, seed, call)
        st.commit(torch.from_numpy(acc).cuda())
        orc.commit(acc[sel], f64s[0], f64s[1], f64s[3])
    assert worst <= TOL, worst
    assert st.status() == 0


def test_bad_accept_sets_status_and_commits_nothing():
    shape = sg.LayerShape(2, 2, 64, 128, 1, "f32")
    st, _, _ = make_store(shape, 13, L=4, T=2)
    devs, _ = draft_device(shape, 13, 0, 2)
    y = torch.empty(2, 2, 2, 64, device="cuda")
    st.verify(2, *devs, y)
    st.commit(torch.tensor([3, 1], dtype=torch.int32, device="cuda"))
    meta = st.region("meta").cpu().numpy()
    assert meta[0, 1] == 0 and meta[1, 1] == 1 and np.all(meta[:, 2] == 0)
    assert st.status(clear=True) == R.REPLAY_DEV_BAD_ACCEPT
    assert st.status() == 0
    st.commit(torch.tensor([1, 0], dtype=torch.int32, device="cuda"))   # nothing pending
    assert st.status() == R.REPLAY_DEV_BAD_ACCEPT


def test_corrupt_metadata_gives_nan_and_status():
    shape = sg.LayerShape(2, 2, 64, 128, 1, "f32")
    st, _, _ = make_store(shape, 14, L=4)
    st.region("meta")[1, 1] = 99                        # beyond the ring
    devs, _ = step_inputs(shape, 14, 0)
    y = torch.zeros(2, 2, 64, device="cuda")
    st.step(*devs, y)
    assert st.status() & R.REPLAY_DEV_BAD_META
    assert torch.isnan(y[1]).all() and not torch.isnan(y[0]).any()


def test_host_errors():
    shape = sg.LayerShape(2, 2, 64, 128, 1, "f32")
    st, _, _ = make_store(shape, 15, L=4, T=2)
    devs, _ = draft_device(shape, 15, 0, 2)
    y = torch.empty(2, 3, 2, 64, device="cuda")
    with pytest.raises(R.ReplayError) as e:
        st.verify(3, *devs, y)
    assert e.value.code == -3
    with pytest.raises(R.ReplayError) as e:
        st.verify(0, *devs, y)
    assert e.value.code == -1


def test_fused_and_split_step_paths_agree():
    """Calls with few slabs take the single fused kernel, larger ones the per-group prep +
    per-head kernels. The same sequences (inputs do not depend on the batch size) through
    both paths -- 128 and 129 sequences x 64 heads straddle the threshold -- agree with each
    other and with the oracle, across two flushes."""
    outs = []
    sel = np.array([0, 63, 127])
    for batch in (128, 129):
        shape = sg.LayerShape(batch, 64, 64, 128, 4, "bf16")
        st, A, D = make_store(shape, 16, L=4)
        orc = Mamba2Decoder(A, D, 4, np.zeros((3, 64, 64, 128)))
        y = torch.empty(batch, 64, 64, device="cuda")
        ys = []
        for t in range(9):
            devs, f64 = step_inputs(shape, 16, t, sel)
            st.step(*devs, y)
            assert rel_vec_err(y[sel].cpu().numpy(), orc.step(*f64), 2).max() <= TOL, (batch, t)
            ys.append(y[:128].cpu().numpy().copy())
        assert st.status() == 0
        outs.append(np.stack(ys))
    assert rel_vec_err(outs[1], outs[0], 3).max() <= 1e-5


@pytest.mark.parametrize("rc,bound", [(R.REPLAY_RC_BF16, 1e-2), (R.REPLAY_RC_FP8E4M3, 0.25),
                                      (R.REPLAY_RC_FP16, 2e-3)])
def test_read_copy_on_the_large_call_path(rc, bound):
    """Above the fused-kernel threshold a read copy is read by CTAs that each take several
    heads of a group (packed copy tiles). 72 sequences x 128 heads, 8 groups, across two
    flushes; the oracle follows three sequences, and the FP32 checkpoints stay exact."""
    shape = sg.LayerShape(72, 128, 64, 128, 8, "bf16")
    wy, wh, _, _ = run_decode(shape, 18, 8, seed=17, read_copy=rc, seqs=[0, 35, 71])
    assert wy <= bound and wh <= TOL, (wy, wh)


class _SrRounder:
    """FP16 stochastic rounding of the followed sequences, one epoch per call (the first
    flush is write number 1; the load or reset was number 0)."""

    def __init__(self, sel, num_slabs):
        self.sel, self.num_slabs, self.epoch = sel, num_slabs, 1

    def __call__(self, h):
        out = F.fp16_sr_round_state(h, self.epoch, self.sel, self.num_slabs)
        self.epoch += 1
        return out


def _decoded_copy(st, rc, h32):
    """The values a non-flush step reads from the copy of FP32 states h32 [b, H, P, N]."""
    if rc == R.REPLAY_RC_BF16:
        return F.bf16_decode(F.bf16_encode(h32)).astype(np.float64)
    if rc == R.REPLAY_RC_FP16:
        return F.fp16_decode(F.fp16_encode(h32))
    out = np.empty(h32.shape)
    for i in np.ndindex(*h32.shape[:2]):
        qc, sc = F.fp8_slab_quantize(h32[i])
        out[i] = F.fp8_slab_dequantize(qc, sc)
    return out


_BF, _F16, _E4 = R.REPLAY_RC_BF16, R.REPLAY_RC_FP16, R.REPLAY_RC_FP8E4M3


@pytest.mark.parametrize("rc,batch,heads,groups,dtype,dstate", [
    (_BF, 4, 8, 2, "f32", 128), (_F16, 4, 8, 2, "f32", 128), (_E4, 4, 8, 2, "f32", 128),
    (_BF, 72, 128, 8, "bf16", 128), (_F16, 72, 128, 8, "bf16", 128), (_E4, 72, 128, 8, "bf16", 128),
    (_BF, 40, 32, 4, "bf16", 64), (_F16, 40, 32, 4, "f32", 64), (_E4, 40, 32, 4, "bf16", 64),
    (_BF, 40, 32, 4, "f32", 256), (_E4, 40, 32, 4, "bf16", 256),
    (_BF, 17, 64, 8, "bf16", 128), (_E4, 17, 64, 8, "f32", 128), (_F16, 19, 56, 7, "bf16", 128)])
def test_copy_reads_follow_the_decoded_copy(rc, batch, heads, groups, dtype, dstate):
    """Non-flush outputs against the unrolled window evaluated in FP64 from the copy's own
    values (the format's decoding of the loaded FP32 state), within 1e-4: the copy is read
    exactly, whichever kernel reads it. Small calls take the fused kernel; calls of more than
    1024 slabs take the bulk-copy several-heads kernel (2 heads per CTA at dstate 128, 4 at
    64, 2 for E4M3 at 256; here also group sizes of 7 and 8 heads) or, for a bf16 copy at
    dstate 256, the one-head-per-CTA kernel."""
    shape = sg.LayerShape(batch, heads, 64, dstate, groups, dtype)
    L, seed = 8, 31
    st, A, D = make_store(shape, seed, L=L, read_copy=rc)
    sel = np.array([0, batch - 1])
    h0 = sg.initial_state(shape, seed)
    st.load_state(torch.from_numpy(h0).cuda())
    hread = _decoded_copy(st, rc, h0[sel])
    y = torch.empty(batch, heads, 64, device="cuda")
    rec = {k: [] for k in ("x", "B", "dt")}
    worst = 0.0
    for t in range(L - 1):
        devs, f64 = step_inputs(shape, seed, t, sel)
        st.step(*devs, y)
        for k, v in zip(("x", "B", "dt"), (f64[0], f64[1], f64[3])):
            rec[k].append(v)
        ywin = window_output(hread, np.stack(rec["x"], 1), np.stack(rec["B"], 1), np.stack(rec["dt"], 1),
                             f64[2], A, D)
        worst = max(worst, rel_vec_err(y[sel].cpu().numpy(), ywin, 2).max())
    assert worst <= TOL, worst
    assert st.status() == 0


@pytest.mark.parametrize("rc,dtype", [(_E4, "f32"), (_E4, "bf16"), (R.REPLAY_RC_NVFP4, "bf16")])
def test_copy_reads_with_64_buffered_records(rc, dtype):
    """Non-flush reads of an E4M3 or NVFP4 copy with up to 63 buffered records (L = 64: the
    largest record staging of the copy-read kernels) against the unrolled window evaluated in
    FP64 from the copy's own values, within 1e-4 (72 sequences x 128 heads, 8 groups)."""
    shape = sg.LayerShape(72, 128, 64, 128, 8, dtype)
    L, seed = 64, 29
    st, A, D = make_store(shape, seed, L=L, read_copy=rc)
    sel = np.array([0, 71])
    h0 = sg.initial_state(shape, seed)
    st.load_state(torch.from_numpy(h0).cuda())
    hread = F.nvfp4_round_state(h0[sel]) if rc == R.REPLAY_RC_NVFP4 else _decoded_copy(st, rc, h0[sel])
    y = torch.empty(72, 128, 64, device="cuda")
    rec = {k: [] for k in ("x", "B", "dt")}
    worst = 0.0
    for t in range(L - 1):
        devs, f64 = step_inputs(shape, seed, t, sel)
        st.step(*devs, y)
        for k, v in zip(("x", "B", "dt"), (f64[0], f64[1], f64[3])):
            rec[k].append(v)
        if t % 7 == 6 or t >= L - 3:
            ywin = window_output(hread, np.stack(rec["x"], 1), np.stack(rec["B"], 1), np.stack(rec["dt"], 1),
                                 f64[2], A, D)
            worst = max(worst, rel_vec_err(y[sel].cpu().numpy(), ywin, 2).max())
    assert worst <= TOL, worst
    assert st.status() == 0


def test_e4m3_reads_at_extreme_query_scales():
    """The E4M3 copy read at dstate 128 splits each group's C into E4M3 terms under a power-of-two
    scale taken from max |C|. Groups whose C is scaled by 1, 0, 1e-30, 1e30, 1e-20, 1e20, or has
    one column 1e3 above the rest, still give the decoded copy's outputs within 1e-4 (FP32
    inputs; 17 sequences x 64 heads, 8 groups: the large-call path)."""
    shape = sg.LayerShape(17, 64, 64, 128, 8, "f32")
    L, seed = 8, 33
    st, A, D = make_store(shape, seed, L=L, read_copy=R.REPLAY_RC_FP8E4M3)
    sel = np.array([0, 9, 16])
    h0 = sg.initial_state(shape, seed)
    st.load_state(torch.from_numpy(h0).cuda())
    hread = _decoded_copy(st, R.REPLAY_RC_FP8E4M3, h0[sel])
    scale = np.array([1.0, 0.0, 1e-30, 1e30, 1.0, 1e-20, 1e20, 1.0], dtype=np.float32)
    y = torch.empty(17, 64, 64, device="cuda")
    rec = {k: [] for k in ("x", "B", "dt")}
    worst = 0.0
    for t in range(L - 1):
        d = sg.token_inputs(shape, seed, [t])
        c32 = np.ascontiguousarray(d["C"].store[:, 0]).astype(np.float32) * scale[None, :, None]
        c32[:, 4, 5] *= np.float32(1e3)  # group 4: one column far above the others
        devs = [torch.from_numpy(np.ascontiguousarray(d[k].store[:, 0])).cuda() for k in ("x", "B")]
        devs += [torch.from_numpy(c32).cuda(), torch.from_numpy(np.ascontiguousarray(d["dt"].store[:, 0])).cuda()]
        st.step(*devs, y)
        for k in ("x", "B", "dt"):
            rec[k].append(d[k].f64[sel, 0])
        ywin = window_output(hread, np.stack(rec["x"], 1), np.stack(rec["B"], 1), np.stack(rec["dt"], 1),
                             c32[sel].astype(np.float64), A, D)
        worst = max(worst, rel_vec_err(y[sel].cpu().numpy(), ywin, 2).max())
    assert worst <= TOL, worst
    assert st.status() == 0


@pytest.mark.parametrize("rc,tol", [(R.REPLAY_RC_BF16, 5e-3), (R.REPLAY_RC_FP8E4M3, 5e-2),
                                    (R.REPLAY_RC_FP16, 1e-3), (R.REPLAY_RC_NVFP4, 5e-2)])
@pytest.mark.parametrize("batch,heads,groups", [(4, 8, 2), (72, 128, 8)])
def test_shared_checkpoint_matches_periodic_rounding(rc, tol, batch, heads, groups):
    """With shared_checkpoint the low-precision copy is the recurrence state: every flush
    starts from it and writes only it. The oracle rounds its FP64 state the same way after
    every L-th token (FP16: stochastically, with the same draws). Outputs follow that oracle
    (up to rare rounding flips between FP32 and FP64 states) and drift from the unrounded
    one."""
    shape = sg.LayerShape(batch, heads, 64, 128, groups, "f32")
    L, steps, seed = 8, 40, 18
    A, D = sg.head_params(heads, seed)
    cfg = R.ReplayConfig(batch, heads, 64, 128, groups, L, 0, R.REPLAY_F32, rc, 1)
    st = R.ReplayStore(cfg, torch.from_numpy(A), torch.from_numpy(D))
    sel = np.array([0, batch - 1])
    rounder = {R.REPLAY_RC_BF16: F.bf16_round_state, R.REPLAY_RC_FP8E4M3: F.e4m3_round_state,
               R.REPLAY_RC_FP16: _SrRounder(sel, batch * heads), R.REPLAY_RC_NVFP4: F.nvfp4_round_state}[rc]
    z = np.zeros((2, heads, 64, 128))
    rounded = Mamba2Decoder(A.astype(float), D.astype(float), groups, z, window_round=rounder, window_L=L)
    plain = Mamba2Decoder(A.astype(float), D.astype(float), groups, z)
    y = torch.empty(batch, heads, 64, device="cuda")
    e_round = e_plain = 0.0
    for t in range(steps):
        devs, f64 = step_inputs(shape, seed, t, sel)
        st.step(*devs, y)
        yg = y[sel].cpu().numpy()
        e_round = max(e_round, rel_vec_err(yg, rounded.step(*f64), 2).max())
        e_plain = max(e_plain, rel_vec_err(yg, plain.step(*f64), 2).max())
    h = torch.empty(batch, heads, 64, 128, device="cuda")
    st.export_state(h)                     # the last step was a flush: h is the stored copy
    hg = h.cpu().numpy()
    # The checkpoint is the rounded state itself: every value lies on the format's grid.
    if rc == R.REPLAY_RC_BF16:
        assert not np.any(hg.view(np.uint32) & 0xFFFF)
    elif rc == R.REPLAY_RC_FP16:
        assert np.array_equal(hg, hg.astype(np.float16).astype(np.float32))
    elif rc == R.REPLAY_RC_NVFP4:
        q = device_codes(st.region("rc").cpu().numpy())
        sb, sgl = st.region("bscale").cpu().numpy(), st.region("scale").cpu().numpy()
        for i in sel:
            for hh in range(heads):
                back = F.nvfp4_slab_dequantize(q[i, hh], sb[i, hh], sgl[i, hh]).astype(np.float32)
                assert np.array_equal(back, hg[i, hh]), (i, hh)
    else:
        scale = st.region("scale").cpu().numpy()[:, :, None, None]
        assert np.array_equal(F.fp8_slab_dequantize(F.e4m3_encode(hg / scale), scale), hg)
    # ... and follows the rounded oracle. FP32 and FP64 states can round a value that sits
    # near a midpoint (or a scale) differently: such flips move one element by one code
    # step and are rare; everything else agrees to FP32 accuracy.
    step = {R.REPLAY_RC_BF16: 2.0 ** -7, R.REPLAY_RC_FP8E4M3: 32 / 448, R.REPLAY_RC_FP16: 2.0 ** -10,
            R.REPLAY_RC_NVFP4: 1 / 3}[rc]
    d = np.abs(hg[sel] - rounded.h) / np.abs(rounded.h).max(axis=(2, 3), keepdims=True)
    assert d.max() <= 2 * step and (d > 1e-5).mean() <= 1e-3, (d.max(), (d > 1e-5).mean())
    assert e_round <= tol and e_plain > 2 * e_round, (e_round, e_plain)
    assert st.status() == 0


def _decoded_nvfp4(st, seqs):
    """The values non-flush steps read from the store's NVFP4 copy, decoded from the device's
    own codes, block scales and slab scales by the oracle's decoder."""
    q = device_codes(st.region("rc").cpu().numpy()[seqs])
    sb, sgl = st.region("bscale").cpu().numpy()[seqs], st.region("scale").cpu().numpy()[seqs]
    out = np.empty(q.shape)
    for i in np.ndindex(*q.shape[:2]):
        out[i] = F.nvfp4_slab_dequantize(q[i], sb[i], sgl[i])
    return out


def _device_copy(st, rc, seqs):
    """The values non-flush steps read from the store's read copy, decoded from the device's
    own bytes (and scales) by the oracle's decoders."""
    if rc == R.REPLAY_RC_NVFP4:
        return _decoded_nvfp4(st, seqs)
    if rc == R.REPLAY_RC_BF16:
        return st.region("rc")[seqs].float().cpu().numpy().astype(np.float64)
    codes = st.region("rc").cpu().numpy()[seqs]
    sc = st.region("scale").cpu().numpy()[seqs].astype(np.float32)
    return (F.e4m3_decode(codes).astype(np.float32) * sc[:, :, None, None]).astype(np.float64)


def _round_copy(rc, h32):
    """The read copy the format gives the FP32 states h32 [b, H, P, N], read back."""
    if rc == R.REPLAY_RC_NVFP4:
        return F.nvfp4_round_state(h32)
    if rc == R.REPLAY_RC_BF16:
        return F.bf16_round_state(h32)
    return F.e4m3_round_state(h32)


@pytest.mark.parametrize("batch,heads,groups,dtype,rc", [
    (4, 8, 2, "f32", R.REPLAY_RC_NVFP4), (72, 128, 8, "bf16", R.REPLAY_RC_NVFP4),
    (72, 128, 8, "bf16", R.REPLAY_RC_BF16), (72, 128, 8, "f32", R.REPLAY_RC_FP8E4M3),
    (4, 8, 2, "bf16", R.REPLAY_RC_FP8E4M3)])
def test_fp16_sr_checkpoint_with_nvfp4_reads(batch, heads, groups, dtype, rc):
    """The recurrence checkpoint in FP16 with stochastic rounding, and a separate read copy
    (NVFP4, bf16 or E4M3) cast from the same FP32 fold (post, "Benefit 3": NVFP4 reads with an
    FP16 recurrence). Checked: flush outputs and the FP16 checkpoints follow the oracle that
    rounds its state stochastically after every window, with the same draws (up to rare flips
    between FP32 and FP64 states); non-flush outputs equal the window evaluated in FP64 from the
    device's decoded copy, within 1e-4; the copy is the encoding of the flush's unrounded state
    (up to the same rare flips), not of the FP16 checkpoint."""
    shape = sg.LayerShape(batch, heads, 64, 128, groups, dtype)
    L, steps, seed = 8, 24, 27
    A, D = sg.head_params(heads, seed)
    cfg = R.ReplayConfig(batch, heads, 64, 128, groups, L, 0, DTYPE[dtype], rc, 0, R.REPLAY_CKPT_F16_SR)
    st = R.ReplayStore(cfg, torch.from_numpy(A), torch.from_numpy(D))
    sel = np.array([0, batch - 1])
    A64, D64 = A.astype(float), D.astype(float)
    z = np.zeros((2, heads, 64, 128))
    rounded = Mamba2Decoder(A64, D64, groups, z, window_round=_SrRounder(sel, batch * heads), window_L=L)
    pre = Mamba2Decoder(A64, D64, groups, z.copy())       # the unrounded state within a window
    y = torch.empty(batch, heads, 64, device="cuda")
    rec = {k: [] for k in ("x", "B", "dt")}
    hread = np.zeros((2, heads, 64, 128))
    e_read = e_flush = 0.0
    for t in range(steps):
        devs, f64 = step_inputs(shape, seed, t, sel)
        st.step(*devs, y)
        yr = rounded.step(*f64)
        pre.step(*f64)
        yg = y[sel].cpu().numpy()
        for k, v in zip(("x", "B", "dt"), (f64[0], f64[1], f64[3])):
            rec[k].append(v)
        if (t + 1) % L:
            ywin = window_output(hread, np.stack(rec["x"], 1), np.stack(rec["B"], 1), np.stack(rec["dt"], 1),
                                 f64[2], A64, D64)
            e_read = max(e_read, rel_vec_err(yg, ywin, 2).max())
            continue
        e_flush = max(e_flush, rel_vec_err(yg, yr, 2).max())
        h16 = st.region("h0").float().cpu().numpy()[sel]
        d = np.abs(h16 - rounded.h) / np.abs(rounded.h).max(axis=(2, 3), keepdims=True)
        assert d.max() <= 2 * 2.0 ** -10 and (d > 1e-5).mean() <= 1e-3, (t, d.max(), (d > 1e-5).mean())
        hread = _device_copy(st, rc, sel)
        want = np.stack([_round_copy(rc, pre.h[i:i + 1])[0] for i in range(2)])
        flips = np.abs(hread - want) > 1e-6 * np.abs(want).max()
        assert flips.mean() <= 1e-3, (t, flips.mean())
        from_ckpt = _round_copy(rc, h16)
        assert np.abs(hread - from_ckpt).max() > 0                 # cast from FP32, not from FP16
        pre = Mamba2Decoder(A64, D64, groups, rounded.h.copy())   # the next window starts from it
        rec = {k: [] for k in ("x", "B", "dt")}
    assert e_read <= TOL and e_flush <= 1e-3, (e_read, e_flush)
    assert st.status() == 0
