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
