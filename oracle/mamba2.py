"""Plain FP64 Mamba-2 decode recurrence and its unrolled (replay) forms.

TEST INFRASTRUCTURE ONLY (see the package docstring): slow, obviously correct, no
blocking, fusion or reordering beyond what each definition states.

Notation (per sequence b and head h; head h belongs to group h // (H / G), heads of a
group being contiguous, the Mamba-2 convention):

    a_t = exp(dt_t * A_h)                    A_h < 0, dt_t > 0 scalars
    h_t = a_t * h_{t-1} + dt_t * x_t B_t^T   h in R^{P x N}, x_t in R^P, B_t, C_t in R^N
    y_t = h_t C_t + D_h * x_t

Source: "ReplaySSM: Rethinking State Storage for Faster Hybrid-Model Decoding" (NVIDIA
Developer blog), section "Why SSM layers can become a decoding bottleneck". The
displayed recurrence was lost in extraction; the text around it fixes its parts: a
data-dependent decay, a rank-1 (outer-product) update, an output read with C, and a
state stored back. The form above is the standard Mamba-2 decode step with exactly those
parts and no more (no dt bias, gate, convolution or norm).

Shapes used throughout: ``h[b, H, P, N]``, ``x[b, H, P]``, ``B, C[b, G, N]``,
``dt[b, H]``, ``A, D[H]``. Multi-token tensors put the token axis second:
``xs[b, k, H, P]``, ``Bs[b, k, G, N]``, ``dts[b, k, H]``.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "group_of_head", "update_state", "read_output", "decode_step", "Mamba2Decoder",
    "window_state", "window_output", "draft_outputs",
]


def group_of_head(nheads: int, ngroups: int) -> np.ndarray:
    """Group index of each head: heads are contiguous per group."""
    return np.arange(nheads) // (nheads // ngroups)


def _per_head(v: np.ndarray, nheads: int) -> np.ndarray:
    """Spread a per-group tensor ``[b, G, N]`` to per-head ``[b, H, N]``."""
    return v[:, group_of_head(nheads, v.shape[1]), :]


def update_state(h, x, B, dt, A):
    """State update: h <- exp(dt * A) * h + dt * x B^T (decay plus rank-1 update)."""
    H = x.shape[1]
    decay = np.exp(dt * A[None, :])                                   # [b, H]
    rank1 = (dt[:, :, None] * x)[:, :, :, None] * _per_head(B, H)[:, :, None, :]
    return decay[:, :, None, None] * h + rank1


def read_output(h, C, x, D):
    """Output read: y = h C + D * x."""
    H = x.shape[1]
    return np.einsum("bhpn,bhn->bhp", h, _per_head(C, H)) + D[None, :, None] * x


def decode_step(h, x, B, C, dt, A, D):
    """One conventional decode step: load, decay + rank-1 update, read with C.

    Returns ``(h_next, y)``; ``h`` is not modified.
    """
    h_next = update_state(h, x, B, dt, A)
    return h_next, read_output(h_next, C, x, D)


class Mamba2Decoder:
    """Step-by-step FP64 decoder for a batch of sequences, with speculative drafts.

    ``verify`` runs drafts forward from the committed state without keeping the result;
    ``commit`` advances each sequence over exactly its first ``accept[b]`` drafts by
    decoding them again. Source: the blog post's section "Benefit 2: Simplify rollback
    and speed up verification" -- outputs are those of decoding the accepted prefix.
    """

    def __init__(self, A, D, ngroups: int, h0, window_round=None, window_L=None):
        """``window_round`` (optional, with ``window_L``): a low-precision checkpoint that is
        also the recurrence state. After every ``window_L``-th decode step the state is
        replaced by ``window_round(state)`` -- the periodic checkpoint of the blog post's
        section "Benefit 3" (rounded once every L steps, and fed back); the output of that
        step is read before the rounding."""
        self.A = np.asarray(A, dtype=np.float64)
        self.D = np.asarray(D, dtype=np.float64)
        self.ngroups = ngroups
        self.h = np.array(h0, dtype=np.float64, copy=True)
        self.window_round, self.window_L, self.t = window_round, window_L, 0

    def step(self, x, B, C, dt):
        self.h, y = decode_step(self.h, x, B, C, dt, self.A, self.D)
        self.t += 1
        if self.window_round is not None and self.t % self.window_L == 0:
            self.h = self.window_round(self.h)
        return y

    def verify(self, xs, Bs, Cs, dts):
        """Outputs ``y[b, T, H, P]`` of T drafts decoded in order; state unchanged."""
        h = self.h
        ys = []
        for j in range(xs.shape[1]):
            h, y = decode_step(h, xs[:, j], Bs[:, j], Cs[:, j], dts[:, j], self.A, self.D)
            ys.append(y)
        return np.stack(ys, axis=1)

    def commit(self, accept, xs, Bs, dts):
        """Advance sequence b over its first ``accept[b]`` drafts (0 <= a <= T)."""
        accept = np.asarray(accept)
        for j in range(xs.shape[1]):
            h_next = update_state(self.h, xs[:, j], Bs[:, j], dts[:, j], self.A)
            take = (j < accept)[:, None, None, None]
            self.h = np.where(take, h_next, self.h)


def _suffix_decay(dts, A, k):
    """gamma[b, s, H] = exp(A * sum_{r=s+1..k} dt_r) for s = 1..k (index s-1), and
    Gamma[b, H] = exp(A * sum_{r=1..k} dt_r); sums taken directly over each range."""
    b, _, H = dts.shape
    gamma = np.empty((b, k, H))
    for s in range(1, k + 1):
        gamma[:, s - 1, :] = np.exp(A[None, :] * dts[:, s:k, :].sum(axis=1))
    Gamma = np.exp(A[None, :] * dts[:, 0:k, :].sum(axis=1))
    return gamma, Gamma


def window_state(h0, xs, Bs, dts, A):
    """The recurrence unrolled over a window of k records (the checkpoint + buffer form).

        h_k = Gamma_k * h0 + sum_{s=1..k} gamma(k, s) * dt_s * x_s B_s^T
        gamma(k, s) = exp(A * sum_{r=s+1..k} dt_r)   (gamma(k, k) = 1)
        Gamma_k     = exp(A * sum_{r=1..k} dt_r)     (the cumulative decay)

    Source: the blog post's section "How ReplaySSM represents the state": the state
    before the window times the cumulative decay, plus the buffered records (x, B, dt).
    The displayed equation was lost; this is the recurrence unrolled by induction.
    This is also what a flush writes as the new checkpoint.
    """
    k = xs.shape[1]
    H = xs.shape[2]
    gamma, Gamma = _suffix_decay(dts, A, k)
    h = Gamma[:, :, None, None] * h0
    for s in range(k):
        w = gamma[:, s, :] * dts[:, s, :]                                      # [b, H]
        h = h + (w[:, :, None] * xs[:, s])[:, :, :, None] * _per_head(Bs[:, s], H)[:, :, None, :]
    return h


def window_output(h0, xs, Bs, dts, C, A, D):
    """Output of the k-th record of a window, computed without building the state.

        y_k = Gamma_k * (h0 C) + sum_{s=1..k} gamma(k, s) * dt_s * (B_s . C) * x_s + D * x_k

    Source: the blog post's sections "How ReplaySSM represents the state" (a non-flush
    step computes the output from checkpoint and buffer) and "Benefit 2" (output-only
    evaluation: dt x B^T read with C equals the scalar dt (B . C) times the vector x).
    """
    k = xs.shape[1]
    H = xs.shape[2]
    gamma, Gamma = _suffix_decay(dts, A, k)
    Ch = _per_head(C, H)
    y = Gamma[:, :, None] * np.einsum("bhpn,bhn->bhp", h0, Ch)
    for s in range(k):
        bc = np.einsum("bhn,bhn->bh", _per_head(Bs[:, s], H), Ch)
        y = y + (gamma[:, s, :] * dts[:, s, :] * bc)[:, :, None] * xs[:, s]
    return y + D[None, :, None] * xs[:, k - 1]


def draft_outputs(h0, rec, drafts, A, D):
    """Output-only evaluation of T drafts against n committed records, in matrix form.

    For each (sequence, head), with the records and drafts numbered s = 1..n+T:

        Q = C of the drafts          [T, N]    (shared by the heads of a group)
        K = B of records and drafts  [n+T, N]  (shared by the heads of a group)
        V_s = dt_s * x_s             [n+T, P]
        M[j, s] = gamma(n+j, s) if s <= n+j else 0     (causally masked decays)
        G_j = Gamma_{n+j}                               (cumulative decay of draft j)
        Y = diag(G) (Q h0^T) + (M o (Q K^T)) V + D * X_drafts

    Source: the blog post's section "Benefit 2: Simplify rollback and speed up
    verification". The expression itself was lost in extraction; the text names its
    parts (cumulative decays of the draft positions, a causally masked decay matrix, two
    small matrix products over cached keys, cached values and draft queries, a term
    shared by the heads of a group). This is the chunkwise form with those parts.

    ``rec`` = (xs, Bs, dts) of the n committed records (n may be 0); ``drafts`` =
    (xs, Bs, Cs, dts) of the T drafts. Returns ``y[b, T, H, P]``.
    """
    xr, Br, dr = rec
    xd, Bd, Cd, dd = drafts
    n, T = xr.shape[1], xd.shape[1]
    H = xd.shape[2]
    grp = group_of_head(H, Bd.shape[2])
    X = np.concatenate([xr, xd], axis=1)                 # [b, n+T, H, P]
    Kb = np.concatenate([Br, Bd], axis=1)[:, :, grp, :]  # [b, n+T, H, N]
    dt = np.concatenate([dr, dd], axis=1)                # [b, n+T, H]
    Q = Cd[:, :, grp, :]                                 # [b, T, H, N]
    V = dt[:, :, :, None] * X                            # [b, n+T, H, P]
    bsz = X.shape[0]
    M = np.zeros((bsz, T, n + T, H))
    G = np.empty((bsz, T, H))
    for j in range(1, T + 1):
        k = n + j
        for s in range(1, k + 1):
            M[:, j - 1, s - 1, :] = np.exp(A[None, :] * dt[:, s:k, :].sum(axis=1))
        G[:, j - 1, :] = np.exp(A[None, :] * dt[:, 0:k, :].sum(axis=1))
    QK = np.einsum("bjhn,bshn->bjsh", Q, Kb)
    Y = G[:, :, :, None] * np.einsum("bhpn,bjhn->bjhp", h0, Q)
    Y = Y + np.einsum("bjsh,bshp->bjhp", M * QK, V)
    return Y + D[None, None, :, None] * xd
