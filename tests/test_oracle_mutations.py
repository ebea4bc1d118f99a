"""Plant plausible mistakes in the oracle (CPU only) and check that the pins catch each.

A pin suite that still passed with one of these mistakes would not pin the oracle.
"""
import numpy as np
import pytest

import oracle.mamba2 as m2
from oracle_pins import ALL_PINS


def _fails_some_pin():
    for pin in ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            return pin.__name__
    return None


def _drop_skip(h, C, x, D):
    return np.einsum("bhpn,bhn->bhp", h, m2._per_head(C, x.shape[1]))


def _decay_sign(h, x, B, dt, A):
    return m2.update_state.__wrapped__(h, x, B, dt, -A)


def _transposed(h, x, B, dt, A):
    H = x.shape[1]
    decay = np.exp(dt * A[None, :])
    Bh = m2._per_head(B, H)
    rank1 = (dt[:, :, None] * Bh)[:, :, :, None] * x[:, :, None, :]   # B x^T instead of x B^T
    return decay[:, :, None, None] * h + rank1


def _no_dt_in_update(h, x, B, dt, A):
    H = x.shape[1]
    decay = np.exp(dt * A[None, :])
    return decay[:, :, None, None] * h + x[:, :, :, None] * m2._per_head(B, H)[:, :, None, :]


def _interleaved_groups(nheads, ngroups):
    return np.arange(nheads) % ngroups


def _gamma_off_by_one(dts, A, k):
    b, _, H = dts.shape
    gamma = np.empty((b, k, H))
    for s in range(1, k + 1):
        gamma[:, s - 1, :] = np.exp(A[None, :] * dts[:, s - 1:k, :].sum(axis=1))
    return gamma, np.exp(A[None, :] * dts[:, 0:k, :].sum(axis=1))


def _commit_one_more(self, accept, xs, Bs, dts):
    accept = np.asarray(accept) + 1
    for j in range(xs.shape[1]):
        h_next = m2.update_state(self.h, xs[:, j], Bs[:, j], dts[:, j], self.A)
        self.h = np.where((j < accept)[:, None, None, None], h_next, self.h)


MUTATIONS = {
    "drop_D_skip": ("read_output", _drop_skip),
    "decay_sign_flipped": ("update_state", _decay_sign),
    "outer_product_transposed": ("update_state", _transposed),
    "dt_missing_from_update": ("update_state", _no_dt_in_update),
    "groups_interleaved": ("group_of_head", _interleaved_groups),
    "gamma_off_by_one": ("_suffix_decay", _gamma_off_by_one),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    orig = getattr(m2, attr)
    fn.__wrapped__ = orig
    monkeypatch.setattr(m2, attr, fn)
    assert _fails_some_pin() is not None, f"no pin catches {name}"


def test_commit_off_by_one_is_caught(monkeypatch):
    monkeypatch.setattr(m2.Mamba2Decoder, "commit", _commit_one_more)
    assert _fails_some_pin() is not None


def test_unmutated_oracle_passes_all_pins():
    assert _fails_some_pin() is None


# ------------------------------------------------------------------ storage formats
import oracle.formats as fm  # noqa: E402
import test_oracle_formats as fmt_pins  # noqa: E402

FORMAT_PINS = [getattr(fmt_pins, n) for n in dir(fmt_pins) if n.startswith("test_")]


def _format_pin_fails():
    for pin in FORMAT_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            return pin.__name__
    return None


def _e2m1_ties_away(v):
    f = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(f)
    d = np.abs(a[..., None] - fm._E2M1_POS)
    code = np.where(d == d.min(axis=-1, keepdims=True), np.arange(8), -1).max(axis=-1)   # larger on ties
    return (code | np.where(np.signbit(f), 0x8, 0)).astype(np.uint8)


def _pack_swapped(q):
    q = np.asarray(q, dtype=np.uint8)
    return ((q[..., 0::2] & 0xF) << 4) | (q[..., 1::2] & 0xF)


def _slab_scale_without_e2m1_max(h):
    h = np.asarray(h, dtype=np.float32)
    P, N = h.shape
    absmax = np.float32(np.max(np.abs(h)))
    s_g = np.float32(1.0) if absmax == 0 else np.float32(absmax / np.float32(fm.E4M3_MAX))
    blocks = h.reshape(P, N // 16, 16)
    s_b = fm.e4m3_encode((np.max(np.abs(blocks), axis=2) / (np.float32(6.0) * s_g)).astype(np.float32))
    e = (fm.e4m3_decode(s_b).astype(np.float32) * s_g).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(e[:, :, None] > 0, fm.e2m1_encode((blocks / e[:, :, None]).astype(np.float32)), 0)
    return q.reshape(P, N).astype(np.uint8), s_b, s_g


def _sr_round_to_nearest(v, u):
    return fm.fp16_encode(v)


def _sr_state(index_of):
    """fp16_sr_round_state with the draw index computed by index_of(epoch, slab, num_slabs, elem)."""
    def rounded(h, epoch, slabs, num_slabs):
        h32 = np.asarray(h, dtype=np.float64).astype(np.float32)
        bsz, H, P, N = h32.shape
        slab = (np.asarray(slabs, dtype=np.uint64).reshape(-1, 1) * np.uint64(H) +
                np.arange(H, dtype=np.uint64).reshape(1, -1)).reshape(bsz, H, 1, 1)
        elem = np.arange(P * N, dtype=np.uint64).reshape(1, 1, P, N)
        idx = index_of(np.uint64(epoch), slab, np.uint64(num_slabs), np.uint64(P * N), elem, bsz, H)
        return fm.fp16_decode(fm.fp16_sr_encode(h32, fm.sr_uniform(idx)))
    return rounded


def _sr_local_slab(e, s, n, pn, elem, bsz, H):      # slabs numbered within the followed subset
    local = (np.arange(bsz, dtype=np.uint64).reshape(-1, 1) * np.uint64(H) +
             np.arange(H, dtype=np.uint64).reshape(1, -1)).reshape(bsz, H, 1, 1)
    return (e * n + local) * pn + elem


def _sr_chunks_low_first(idx):
    idx = np.asarray(idx, dtype=np.uint64)
    z = fm.splitmix64(fm.SR_SEED, idx // np.uint64(4))
    return ((z >> (np.uint64(16) * (idx % np.uint64(4)))) & np.uint64(0xFFFF)).astype(np.float64) * 2.0 ** -16


def _nvfp4_state_blocks_down_columns(h):
    h32 = np.asarray(h, dtype=np.float64).astype(np.float32)
    out = np.empty(h32.shape, dtype=np.float64)
    for idx in np.ndindex(*h32.shape[:-2]):
        out[idx] = fm.nvfp4_slab_dequantize(*fm.nvfp4_slab_quantize(h32[idx].T)).T
    return out


def _nvfp4_state_one_scale(h):
    h32 = np.asarray(h, dtype=np.float64).astype(np.float32)
    P, N = h32.shape[-2:]
    flat = h32.reshape(-1, N)
    return fm.nvfp4_slab_dequantize(*fm.nvfp4_slab_quantize(flat)).reshape(h32.shape)


FORMAT_MUTATIONS = {
    "e2m1_ties_away_from_zero": ("e2m1_encode", _e2m1_ties_away),
    "nvfp4_nibbles_swapped": ("nvfp4_pack", _pack_swapped),
    "nvfp4_slab_scale_missing_6": ("nvfp4_slab_quantize", _slab_scale_without_e2m1_max),
    "fp16_sr_is_round_to_nearest": ("fp16_sr_encode", _sr_round_to_nearest),
    "sr_index_epoch_and_slab_swapped": (
        "fp16_sr_round_state", _sr_state(lambda e, s, n, pn, elem, bsz, H: (s * n + e) * pn + elem)),
    "sr_index_epoch_off_by_one": (
        "fp16_sr_round_state", _sr_state(lambda e, s, n, pn, elem, bsz, H: ((e + np.uint64(1)) * n + s) * pn + elem)),
    "sr_index_subset_numbering_ignored": ("fp16_sr_round_state", _sr_state(_sr_local_slab)),
    "sr_draw_chunks_low_first": ("sr_uniform", _sr_chunks_low_first),
    "nvfp4_state_blocks_down_columns": ("nvfp4_round_state", _nvfp4_state_blocks_down_columns),
    "nvfp4_state_one_scale_for_all_slabs": ("nvfp4_round_state", _nvfp4_state_one_scale),
}


@pytest.mark.parametrize("name", sorted(FORMAT_MUTATIONS))
def test_planted_format_mistake_is_caught(name, monkeypatch):
    attr, fn = FORMAT_MUTATIONS[name]
    monkeypatch.setattr(fm, attr, fn)
    assert _format_pin_fails() is not None, f"no pin catches {name}"


def test_unmutated_formats_pass_all_pins():
    assert _format_pin_fails() is None
