"""Pins of the KDA oracle against what the pages and the mathematics fix.

Each ``pin_*`` function takes an :class:`oracle.Oracle` and raises
AssertionError when it disagrees with a value that does not come from the
oracle itself: closed forms, invariants, brute force on tiny inputs, the
golden gate points, or the independent NumPy chunkwise form.  They are run
against the real oracle (tests/test_oracle_pins.py) and against deliberately
broken copies of it (tests/test_oracle_mutants.py), which each pin set must
catch.
"""
from __future__ import annotations

import math
import os

import numpy as np

from oracle import chunk_np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GMIN = -5.0  # "Kimi K3 Technical Report - Open Frontier Intelligence", sec. 2.1.1


def _rng(seed):
    return np.random.default_rng(seed)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _rand_inputs(rng, T, H, dk, dv, beta_scale=1.0):
    q = _unit(rng.standard_normal((T, H, dk)))
    k = _unit(rng.standard_normal((T, H, dk)))
    v = rng.standard_normal((T, H, dv))
    z = rng.standard_normal((T, H, dk))
    beta = beta_scale / (1.0 + np.exp(-rng.standard_normal((T, H))))
    A = rng.uniform(-1.0, 1.0, H)
    return q, k, v, z, beta, A


def _close(a, b, rtol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    if a.size == 0:
        return
    scale = max(np.max(np.abs(b)), 1e-300)
    err = np.max(np.abs(a - b)) / scale
    assert err <= rtol, f"{what}: rel err {err:.3e} > {rtol:.1e}"


# --- gate ---------------------------------------------------------------------------------

def pin_gate_points(orc):
    """Golden closed-form gate values (tests/golden/gate_points.txt)."""
    rows = []
    with open(os.path.join(GOLDEN, "gate_points.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append([float(x) for x in line.split()])
    for A, z, g_expected in rows:
        g = orc.gate(np.array([[[z]]]), np.array([A]), GMIN)[0, 0, 0]
        assert abs(g - g_expected) <= 1e-14, f"gate(A={A}, z={z}) = {g}, expected {g_expected}"


def pin_gate_bounds(orc):
    """exp(g) lies in [exp(gmin), 1] and g is non-increasing in z, for A in [-1, 1]."""
    z = np.concatenate([[-np.inf], np.linspace(-60, 60, 241), [np.inf]])
    for A in (-1.0, -0.3, 0.0, 0.5, 1.0):
        g = orc.gate(z.reshape(-1, 1, 1), np.array([A]), GMIN).ravel()
        a = np.exp(g)
        assert np.all(a >= math.exp(GMIN)) and np.all(a <= 1.0), "decay outside [e^gmin, 1]"
        assert np.all(np.diff(g) <= 0.0), "gate not monotone in z"
        assert g[-1] == GMIN and g[0] == 0.0, "gate limits at +-inf"


# --- closed forms and brute force ---------------------------------------------------------

def pin_t1_closed_form(orc):
    """T = 1: S_1 = (I - b k k^T) Diag(exp(g)) S_0 + b k v^T, o = S_1^T q."""
    rng = _rng(1)
    dk, dv = 5, 3
    q, k, v, z, beta, A = _rand_inputs(rng, 1, 1, dk, dv)
    S0 = rng.standard_normal((1, 1, dk, dv))
    g = orc.gate(z, A, GMIN)[0, 0]
    kk, b = k[0, 0], beta[0, 0]
    S1 = (np.eye(dk) - b * np.outer(kk, kk)) @ np.diag(np.exp(g)) @ S0[0, 0] + b * np.outer(kk, v[0, 0])
    out = orc.prefill(q, k, v, z, beta, A, GMIN, S0=S0)
    _close(out["S_final"][0, 0], S1, 1e-13, "T=1 state")
    _close(out["o"][0, 0], S1.T @ q[0, 0], 1e-13, "T=1 output")
    # S0 = 0: o = b (k . q) v
    out0 = orc.prefill(q, k, v, z, beta, A, GMIN)
    _close(out0["o"][0, 0], b * np.dot(kk, q[0, 0]) * v[0, 0], 1e-13, "T=1 output, S0=0")


def pin_matrix_form(orc):
    """Brute force: compose the matrix form of the recurrence over 7 tokens, 2 heads."""
    rng = _rng(2)
    T, H, dk, dv = 7, 2, 4, 3
    q, k, v, z, beta, A = _rand_inputs(rng, T, H, dk, dv)
    S0 = rng.standard_normal((1, H, dk, dv))
    g = orc.gate(z, A, GMIN)
    out = orc.prefill(q, k, v, z, beta, A, GMIN, S0=S0)
    for h in range(H):
        S = S0[0, h].copy()
        for t in range(T):
            M = (np.eye(dk) - beta[t, h] * np.outer(k[t, h], k[t, h])) @ np.diag(np.exp(g[t, h]))
            S = M @ S + beta[t, h] * np.outer(k[t, h], v[t, h])
            _close(out["o"][t, h], S.T @ q[t, h], 1e-12, f"matrix form o[{t},{h}]")
        _close(out["S_final"][0, h], S, 1e-12, f"matrix form S[{h}]")


def pin_worked_example(orc):
    """Two tokens worked by hand (dk = dv = 2).

    S0 = [[1, 2], [3, 4]].  Token 1: k = (1, 0), v = (10, 20), b = 1/2,
    q = (0, 1), z = -inf (no decay).  p = S0^T k = (1, 2); row 0 gains
    b (v - p) = (4.5, 9) -> S1 = [[5.5, 11], [3, 4]]; o1 = S1^T q = (3, 4).
    Token 2: k = (0.6, 0.8), v = (1, -1), b = 1, q = (1, 0), A = 0, z = 0, so
    g = -2.5 in both channels and a = exp(-2.5).  p = a (0.6 (5.5, 11) +
    0.8 (3, 4)) = a (5.7, 9.8); o2 = row 0 of a S1 + k (v - p)^T
    = (0.6 + 2.08 a, -0.6 + 5.12 a).
    """
    a = math.exp(-2.5)
    q = np.array([[[0.0, 1.0]], [[1.0, 0.0]]])
    k = np.array([[[1.0, 0.0]], [[0.6, 0.8]]])
    v = np.array([[[10.0, 20.0]], [[1.0, -1.0]]])
    z = np.array([[[-np.inf, -np.inf]], [[0.0, 0.0]]])
    beta = np.array([[0.5], [1.0]])
    A = np.array([0.0])
    S0 = np.array([[[[1.0, 2.0], [3.0, 4.0]]]])
    out = orc.prefill(q, k, v, z, beta, A, GMIN, S0=S0)
    _close(out["o"][0, 0], [3.0, 4.0], 1e-15, "worked example o1")
    _close(out["o"][1, 0], [0.6 + 2.08 * a, -0.6 + 5.12 * a], 1e-14, "worked example o2")
    S2 = a * np.array([[5.5, 11.0], [3.0, 4.0]]) + np.outer([0.6, 0.8], [1.0 - 5.7 * a, -1.0 - 9.8 * a])
    _close(out["S_final"][0, 0], S2, 1e-14, "worked example S2")


def pin_beta0_cumprod(orc):
    """b = 0: o_t = S0^T (q_t * prod_{m<=t} exp(g_m)) and S_T = Diag(prod exp(g)) S0."""
    rng = _rng(3)
    T, H, dk, dv = 40, 2, 6, 5
    q, k, v, z, beta, A = _rand_inputs(rng, T, H, dk, dv)
    beta[:] = 0.0
    S0 = rng.standard_normal((1, H, dk, dv))
    g = orc.gate(z, A, GMIN)
    cp = np.cumprod(np.exp(g), axis=0)  # [T, H, dk]
    out = orc.prefill(q, k, v, z, beta, A, GMIN, S0=S0)
    for h in range(H):
        expect = (q[:, h] * cp[:, h]) @ S0[0, h]
        _close(out["o"][:, h], expect, 1e-12, "beta=0 output")
        _close(out["S_final"][0, h], cp[-1, h][:, None] * S0[0, h], 1e-12, "beta=0 state")


def pin_gla_closed_form(orc):
    """Without the erase term (gated linear attention reading):
    o_t = S0^T (q_t * e^{G_t}) + sum_{i<=t} b_i (q_t . (k_i * e^{G_t - G_i})) v_i."""
    rng = _rng(4)
    T, H, dk, dv = 30, 1, 5, 4
    q, k, v, z, beta, A = _rand_inputs(rng, T, H, dk, dv)
    S0 = rng.standard_normal((1, H, dk, dv))
    g = orc.gate(z, A, GMIN)[:, 0]
    G = np.cumsum(g, axis=0)
    out = orc.prefill(q, k, v, z, beta, A, GMIN, S0=S0, erase=False)
    for t in range(T):
        expect = S0[0, 0].T @ (q[t, 0] * np.exp(G[t]))
        for i in range(t + 1):
            expect = expect + beta[i, 0] * np.dot(q[t, 0], k[i, 0] * np.exp(G[t] - G[i])) * v[i, 0]
        _close(out["o"][t, 0], expect, 1e-12, f"GLA closed form o[{t}]")


def pin_erase_is_second_order(orc):
    """KDA minus its erase-free form is O(b^2) as b -> 0 (log-log slope 2)."""
    rng = _rng(5)
    T, H, dk, dv = 12, 1, 6, 4
    q, k, v, z, beta, A = _rand_inputs(rng, T, H, dk, dv)
    diffs = []
    for eps in (1e-2, 1e-3):
        b = beta * eps
        d = orc.prefill(q, k, v, z, b, A, GMIN)["o"] - orc.prefill(q, k, v, z, b, A, GMIN,
                                                                     erase=False)["o"]
        diffs.append(np.max(np.abs(d)))
    slope = math.log(diffs[0] / diffs[1]) / math.log(10.0)
    assert abs(slope - 2.0) < 0.05, f"erase term slope {slope:.3f}, expected 2"


def _hadamard(n):
    Hm = np.array([[1.0]])
    while Hm.shape[0] < n:
        Hm = np.block([[Hm, Hm], [Hm, -Hm]])
    return Hm / math.sqrt(n)


def pin_retrieval(orc):
    """b = 1, no decay, S0 = 0, orthonormal keys (Hadamard rows, +-1/8 exact):
    querying k_j after the writes returns v_j exactly; rewriting k_j with v'
    returns v' (overwrite)."""
    rng = _rng(6)
    dk, dv, n = 64, 16, 40
    keys = _hadamard(dk)[rng.permutation(dk)[:n]]
    vals = np.round(rng.standard_normal((n, dv)) * 256) / 256  # few-bit values: exact sums
    v_new = np.round(rng.standard_normal(dv) * 256) / 256
    # n writes, one overwrite of key 3, then n reads with b = 0
    T = 2 * n + 1
    q = np.zeros((T, 1, dk)); k = np.zeros((T, 1, dk)); v = np.zeros((T, 1, dv))
    beta = np.zeros((T, 1)); z = np.full((T, 1, dk), -np.inf)
    k[:n, 0] = keys; v[:n, 0] = vals; beta[:n, 0] = 1.0; q[:n, 0] = keys
    k[n, 0] = keys[3]; v[n, 0] = v_new; beta[n, 0] = 1.0; q[n, 0] = keys[3]
    q[n + 1:, 0] = keys
    out = orc.prefill(q, k, v, z, beta, np.array([0.3]), GMIN)
    expect = vals.copy()
    expect[3] = v_new
    assert np.array_equal(out["o"][n + 1:, 0], expect), "retrieval is not exact"
    assert np.array_equal(out["o"][:n, 0], vals), "read-after-write is not exact"


def pin_decay_floor(orc):
    """z = +inf in every channel: each step decays by exactly e^-5; with b = 0
    the state after T steps is e^{-5T} S0."""
    rng = _rng(7)
    T, dk, dv = 9, 4, 3
    S0 = rng.standard_normal((1, 1, dk, dv))
    z = np.full((T, 1, dk), np.inf)
    q = np.ones((T, 1, dk)); k = np.ones((T, 1, dk)); v = np.ones((T, 1, dv))
    beta = np.zeros((T, 1))
    out = orc.prefill(q, k, v, z, beta, np.array([-0.4]), GMIN, S0=S0)
    _close(out["S_final"][0, 0], math.exp(-5.0 * T) * S0[0, 0], 1e-13, "decay floor")


# --- chunk form, linearity, state passing -------------------------------------------------

def pin_chunk_form(orc):
    """Independent NumPy chunkwise form equals the sequential oracle (incl. snapshots)."""
    rng = _rng(8)
    for T, dk, dv, C in ((1, 4, 4, 64), (63, 8, 4, 64), (64, 16, 8, 64), (65, 8, 16, 64),
                         (130, 16, 16, 64), (50, 8, 8, 16)):
        q, k, v, z, beta, A = _rand_inputs(rng, T, 1, dk, dv)
        S0 = rng.standard_normal((1, 1, dk, dv)) * 0.1
        g = orc.gate(z, A, GMIN)[:, 0]
        o_c, S_c, snaps_c = chunk_np.chunk_forward(q[:, 0], k[:, 0], v[:, 0], g, beta[:, 0],
                                                   S0[0, 0], chunk=C)
        out = orc.prefill(q, k, v, z, beta, A, GMIN, S0=S0, chunk=C, snapshots=True)
        _close(out["o"][:, 0], o_c, 1e-11, f"chunk form o (T={T})")
        _close(out["S_final"][0, 0], S_c, 1e-11, f"chunk form S (T={T})")
        _close(out["snaps"][:, 0], snaps_c, 1e-11, f"chunk form snapshots (T={T})")
        if T >= 2:
            Akk, Tm = chunk_np.ut_transform(k[:min(T, C), 0], g[:min(T, C)], beta[:min(T, C), 0])
            L = Akk.shape[0]
            _close(Tm @ (np.eye(L) + Akk), np.eye(L), 1e-12, "T (I + A_kk) = I")


def pin_linearity(orc):
    """With S0 = 0 the output is linear in V; column j of o and S depends only
    on column j of V and S0 (permuting value channels permutes the outputs)."""
    rng = _rng(9)
    T, H, dk, dv = 70, 2, 8, 6
    q, k, v, z, beta, A = _rand_inputs(rng, T, H, dk, dv)
    v2 = rng.standard_normal(v.shape)
    o1 = orc.prefill(q, k, v, z, beta, A, GMIN)["o"]
    o2 = orc.prefill(q, k, v2, z, beta, A, GMIN)["o"]
    o12 = orc.prefill(q, k, 2.0 * v - 3.0 * v2, z, beta, A, GMIN)["o"]
    _close(o12, 2.0 * o1 - 3.0 * o2, 1e-12, "linearity in V")
    S0 = rng.standard_normal((1, H, dk, dv))
    perm = rng.permutation(dv)
    a = orc.prefill(q, k, v, z, beta, A, GMIN, S0=S0)
    b = orc.prefill(q, k, v[:, :, perm], z, beta, A, GMIN, S0=S0[..., perm])
    _close(b["o"], a["o"][:, :, perm], 1e-13, "value-column permutation (o)")
    _close(b["S_final"], a["S_final"][..., perm], 1e-13, "value-column permutation (S)")


def pin_state_passing(orc):
    """Prefix caching: [0, L) equals [0, 64m) -> snapshot m -> [64m, L); packed
    sequences equal separate runs; n decode steps equal an n-token prefill."""
    rng = _rng(10)
    C, H, dk, dv = 16, 2, 8, 4
    L = 75
    q, k, v, z, beta, A = _rand_inputs(rng, L, H, dk, dv)
    S0 = rng.standard_normal((1, H, dk, dv)) * 0.5
    whole = orc.prefill(q, k, v, z, beta, A, GMIN, S0=S0, chunk=C, snapshots=True)
    assert whole["snaps"].shape[0] == L // C
    for m in (1, 3):
        cut = m * C
        rest = orc.prefill(q[cut:], k[cut:], v[cut:], z[cut:], beta[cut:], A, GMIN,
                           S0=whole["snaps"][m - 1][None], chunk=C)
        _close(rest["o"], whole["o"][cut:], 1e-12, f"resume from snapshot {m} (o)")
        _close(rest["S_final"], whole["S_final"], 1e-12, f"resume from snapshot {m} (S)")
    # packed varlen == separate
    lens = [20, 33, 16]
    cu = np.concatenate([[0], np.cumsum(lens)])
    qs, ks, vs, zs, bs, _ = _rand_inputs(rng, int(cu[-1]), H, dk, dv)
    S0s = rng.standard_normal((3, H, dk, dv))
    packed = orc.prefill(qs, ks, vs, zs, bs, A, GMIN, cu_seqlens=cu, S0=S0s, chunk=C,
                         snapshots=True)
    for s in range(3):
        sl = slice(cu[s], cu[s + 1])
        one = orc.prefill(qs[sl], ks[sl], vs[sl], zs[sl], bs[sl], A, GMIN, S0=S0s[s:s + 1],
                          chunk=C, snapshots=True)
        _close(packed["o"][sl], one["o"], 1e-13, f"packed vs separate o[{s}]")
        _close(packed["S_final"][s], one["S_final"][0], 1e-13, f"packed vs separate S[{s}]")
        off = packed["snap_offsets"]
        _close(packed["snaps"][off[s]:off[s + 1]], one["snaps"], 1e-13, "packed snapshots")
    # decode steps == prefill
    n = 9
    state = np.ascontiguousarray(S0.copy())
    for t in range(n):
        o_t = orc.decode_step(q[t:t + 1], k[t:t + 1], v[t:t + 1], z[t:t + 1], beta[t:t + 1],
                              A, state)
        _close(o_t[0], whole["o"][t], 1e-13, f"decode vs prefill o[{t}]")
    pre = orc.prefill(q[:n], k[:n], v[:n], z[:n], beta[:n], A, GMIN, S0=S0)
    _close(state, pre["S_final"], 1e-13, "decode vs prefill state")


def pin_norm_bound(orc):
    """Unit keys and b in (0, 1): (I - b k k^T) Diag(a) is a contraction, so
    ||S_t||_F <= ||S_{t-1}||_F + b ||k|| ||v|| at every decode step."""
    rng = _rng(11)
    n, H, dk, dv = 3, 2, 8, 8
    state = np.ascontiguousarray(rng.standard_normal((n, H, dk, dv)))
    A = rng.uniform(-1, 1, H)
    prev = np.linalg.norm(state, axis=(2, 3))
    for _ in range(300):
        q, k, v, z, beta, _ = _rand_inputs(rng, n, H, dk, dv)
        orc.decode_step(q, k, v, z, beta, A, state)
        now = np.linalg.norm(state, axis=(2, 3))
        bound = prev + beta * np.linalg.norm(k, axis=-1) * np.linalg.norm(v, axis=-1)
        assert np.all(now <= bound * (1 + 1e-12)), "state norm grew past the contraction bound"
        prev = now
    assert np.all(np.isfinite(state))


ALL_PINS = [
    pin_gate_points, pin_gate_bounds, pin_t1_closed_form, pin_matrix_form, pin_worked_example,
    pin_beta0_cumprod, pin_gla_closed_form, pin_erase_is_second_order, pin_retrieval,
    pin_decay_floor, pin_chunk_form, pin_linearity, pin_state_passing, pin_norm_bound,
]


# --- input pre-ops (L2 norm of q, k rows; sigmoid of beta) -------------------------------

def _pre(pre):
    if pre is None:
        from oracle import preops as pre
    return pre


def pin_preop_l2norm(orc, pre=None):
    """Unit rows by hand (a 3-4-5 triangle, a 2x2x... cube diagonal, a signed
    axis vector), a zero row, and for random rows: unit length, the same
    direction, and no change under a positive rescale of the row."""
    pre = _pre(pre)
    x = np.array([[3.0, 4.0, 0.0, 0.0], [1.0, 1.0, 1.0, 1.0], [0.0, -2.5, 0.0, 0.0],
                  [0.0, 0.0, 0.0, 0.0]])
    want = np.array([[0.6, 0.8, 0.0, 0.0], [0.5, 0.5, 0.5, 0.5], [0.0, -1.0, 0.0, 0.0],
                     [0.0, 0.0, 0.0, 0.0]])
    _close(pre.l2_normalize_rows(x), want, 1e-15, "hand-normalised rows")
    rng = _rng(21)
    r = rng.standard_normal((5, 3, 16)) * rng.uniform(0.1, 30.0, (5, 3, 1))
    u = pre.l2_normalize_rows(r)
    _close(np.sum(u * u, axis=-1), np.ones((5, 3)), 1e-14, "unit length")
    cos = np.sum(u * r, axis=-1) ** 2 / np.sum(r * r, axis=-1)
    _close(cos, np.ones((5, 3)), 1e-14, "same direction (cos^2 = 1)")
    assert np.all(np.sum(u * r, axis=-1) > 0), "direction flipped"
    _close(pre.l2_normalize_rows(r * 7.25), u, 1e-14, "rescale invariance")


def pin_preop_sigmoid(orc, pre=None):
    """Logistic values fixed by logarithms: sigma(0) = 1/2, sigma(ln 3) = 3/4,
    sigma(-ln 3) = 1/4, sigma(ln 9) = 9/10; saturation without overflow; and
    the derivative identity sigma' = sigma (1 - sigma) by central differences."""
    pre = _pre(pre)
    x = np.array([0.0, math.log(3.0), -math.log(3.0), math.log(9.0), 800.0, -800.0])
    want = np.array([0.5, 0.75, 0.25, 0.9, 1.0, 0.0])
    _close(pre.sigmoid(x), want, 1e-15, "sigmoid at log points")
    xs = np.linspace(-6.0, 6.0, 49)
    h = 1e-5
    d = (pre.sigmoid(xs + h) - pre.sigmoid(xs - h)) / (2 * h)
    s = pre.sigmoid(xs)
    _close(d, s * (1 - s), 1e-8, "sigmoid derivative identity")


def pin_preop_prefill_invariance(orc, pre=None):
    """The recurrence on raw inputs after the pre-ops equals the recurrence on
    the unit rows and beta themselves: q, k given with arbitrary positive row
    scales (different for q and k), beta given as its logit."""
    pre = _pre(pre)
    rng = _rng(22)
    T, H, dk, dv = 70, 2, 8, 6
    q, k, v, z, beta, A = _rand_inputs(rng, T, H, dk, dv)
    cq = rng.uniform(0.05, 20.0, (T, H, 1))
    ck = rng.uniform(0.05, 20.0, (T, H, 1))
    logit = np.log(beta / (1.0 - beta))
    q2, k2, b2 = pre.apply(q * cq, k * ck, logit, True, True)
    ref = orc.prefill(q, k, v, z, beta, A)
    got = orc.prefill(q2, k2, v, z, b2, A)
    _close(got["o"], ref["o"], 1e-12, "outputs after the pre-ops")
    _close(got["S_final"], ref["S_final"], 1e-12, "state after the pre-ops")
    # each switch alone leaves the other input untouched
    q3, k3, b3 = pre.apply(q * cq, k * ck, logit, False, True)
    _close(q3, q * cq, 0.0, "q without the norm switch")
    _close(b3, beta, 1e-13, "beta with the sigmoid switch")
    q4, k4, b4 = pre.apply(q * cq, k * ck, logit, True, False)
    _close(k4, k, 1e-14, "k with the norm switch")
    _close(b4, logit, 0.0, "beta without the sigmoid switch")


PREOP_PINS = [pin_preop_l2norm, pin_preop_sigmoid, pin_preop_prefill_invariance]
