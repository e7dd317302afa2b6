"""Chunkwise form of KDA in NumPy fp64: TEST INFRASTRUCTURE ONLY.

A second, independent CPU implementation used to pin the sequential C oracle
(they agree to rounding on tiny inputs) and to document, in plain dense
matrices, the chunkwise-parallel algebra that the fast path relies on.
"Kimi K3 Technical Report - Open Frontier Intelligence", Method (sec. 2.1)
says KDA has a chunkwise-parallel form without printing it; the form below is
derived here from the recurrence

    S_t = (I - b_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + b_t k_t v_t^T,  o_t = S_t^T q_t

for one chunk of rows r = 0..L-1 with inclusive cumulative log-decay
G_r = sum_{m<=r} g_m (a row vector over key channels):

    D[r, i, c]  = exp(G_r[c] - G_i[c])                    (r >= i)
    A_kk[r, i]  = b_r * sum_c k_r[c] k_i[c] D[r, i, c]    (r > i, else 0)
    T           = (I + A_kk)^{-1}
    U           = T diag(b) V,   Wk = T diag(b) (K * exp(G))
    W           = U - Wk S
    P[r, i]     = sum_c q_r[c] k_i[c] D[r, i, c]          (r >= i, else 0)
    O           = (Q * exp(G)) S + P W
    S'          = Diag(exp(G_last)) S + (K * exp(G_last - G))^T W

It works on log-decays g directly (the caller computes them), uses a dense
solve for T and never factorises exp(G_r - G_i) into two exponentials, so it
shares neither code nor numerical scheme with the fast path.
"""
from __future__ import annotations

import numpy as np


def chunk_forward(q, k, v, g, beta, S0=None, chunk=64, erase=True):
    """Run one (sequence, head) through the chunkwise form.

    q, k, g: [T, dk]; v: [T, dv]; beta: [T]; S0: [dk, dv] or None.
    Returns (o [T, dv], S_final [dk, dv], snaps [floor(T/chunk), dk, dv]).
    With erase=False the delta-rule erase term is dropped (A_kk = 0, T = I).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, np.float64, copy=True)
    o = np.zeros((T, dv))
    snaps = []
    for t0 in range(0, T, chunk):
        t1 = min(t0 + chunk, T)
        L = t1 - t0
        Kc, Qc, Vc, bc = k[t0:t1], q[t0:t1], v[t0:t1], beta[t0:t1]
        G = np.cumsum(g[t0:t1], axis=0)  # [L, dk], inclusive
        r_idx = np.arange(L)[:, None]
        i_idx = np.arange(L)[None, :]
        lower_incl = r_idx >= i_idx
        # exponent G_r - G_i only where r >= i (elsewhere -inf -> exp = 0),
        # so no overflow is ever formed.
        diff = np.where(lower_incl[:, :, None], G[:, None, :] - G[None, :, :], -np.inf)
        D = np.exp(diff)  # [L, L, dk]
        KK = np.einsum("rc,ic,ric->ri", Kc, Kc, D)
        QK = np.einsum("rc,ic,ric->ri", Qc, Kc, D)
        if erase:
            Akk = bc[:, None] * np.where(r_idx > i_idx, KK, 0.0)
        else:
            Akk = np.zeros((L, L))
        Tm = np.linalg.solve(np.eye(L) + Akk, np.eye(L))
        eG = np.exp(G)
        U = Tm @ (bc[:, None] * Vc)
        Wk = Tm @ (bc[:, None] * (Kc * eG))
        W = U - Wk @ S if erase else U
        P = np.where(lower_incl, QK, 0.0)
        o[t0:t1] = (Qc * eG) @ S + P @ W
        G_last = G[-1]
        S = np.exp(G_last)[:, None] * S + (Kc * np.exp(G_last[None, :] - G)).T @ W
        if L == chunk:
            snaps.append(S.copy())
    snaps = np.array(snaps) if snaps else np.zeros((0, dk, dv))
    return o, S, snaps


def ut_transform(k, g, beta):
    """Return (A_kk, T) of one chunk, for the identity T (I + A_kk) = I."""
    k = np.asarray(k, np.float64)
    G = np.cumsum(np.asarray(g, np.float64), axis=0)
    L = k.shape[0]
    r_idx = np.arange(L)[:, None]
    i_idx = np.arange(L)[None, :]
    diff = np.where((r_idx > i_idx)[:, :, None], G[:, None, :] - G[None, :, :], -np.inf)
    Akk = np.asarray(beta, np.float64)[:, None] * np.einsum("rc,ic,ric->ri", k, k, np.exp(diff))
    Tm = np.linalg.solve(np.eye(L) + Akk, np.eye(L))
    return Akk, Tm
