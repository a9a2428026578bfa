"""Pins of the CPU oracle to facts the Mamba-3 pages and mathematics fix.

Each test checks the oracle against something other than itself: a closed
form, a textbook special case, an invariant, a golden fixture derived from
the pages, or a different formulation (rotated-real / matrix form / chunked).
Chosen so that a dropped term, a wrong sign or index, or a transposed operand
fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from chunked_numpy import rot, scan_chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_problem(rng, b=1, L=12, H=2, R=2, P=3, N=6, carry=True, h0=True, theta_scale=math.pi):
    x = rng.standard_normal((b, L, H, R, P))
    B = rng.standard_normal((b, L, H, R, N))
    C = rng.standard_normal((b, L, H, R, N))
    dt = np.log1p(np.exp(rng.standard_normal((b, L, H)) - 1.0))
    A = -np.exp(0.5 * rng.standard_normal((b, L, H)))
    lam = 1.0 / (1.0 + np.exp(-rng.standard_normal((b, L, H))))
    theta = rng.uniform(-theta_scale, theta_scale, (b, L, H, N // 2))
    kw = {}
    if h0:
        kw["h0"] = rng.standard_normal((b, H, N, P))
    if carry:
        kw["Bprev"] = rng.standard_normal((b, H, R, N))
        kw["xprev"] = rng.standard_normal((b, H, R, P))
    return (x, B, C, dt, A, lam, theta), kw


def rel(a, b):
    return np.max(np.abs(a - b)) / max(np.sqrt(np.mean(b * b)), 1e-300)


# --- golden fixture: parity by rotation ------------------------------------------

def test_parity_rotation_golden():
    rows = np.loadtxt(os.path.join(GOLDEN, "parity_rotation.txt"))
    bits, expect = rows[:, 0], rows[:, 1]
    L = len(bits)
    one = lambda v: np.full((1, L, 1), v, dtype=float)
    x = np.ones((1, L, 1, 1, 1))
    B = np.zeros((1, L, 1, 1, 2))
    C = np.zeros((1, L, 1, 1, 2))
    C[..., 0] = 1.0
    theta = (math.pi * bits).reshape(1, L, 1, 1)
    h0 = np.array([1.0, 0.0]).reshape(1, 1, 2, 1)
    for lam in (1.0, 0.5):   # with B = 0 the input weights do not matter
        y, h, _, _ = oracle.scan(x, B, C, one(1.0), one(0.0), one(lam), theta, h0=h0)
        np.testing.assert_allclose(y[0, :, 0, 0, 0], expect, atol=1e-12)


# --- convergence order of the exponential-trapezoid rule -------------------------

def _ode_error(lam, dt, a=-0.7, w=1.3, om=2.1, T=2.0, s0=(0.4 + 0.9j)):
    """Integrates S' = (a + i w) S + e^{i om s} on [0, T]; returns |S_K - S(T)|."""
    K = int(round(T / dt))
    c = a + 1j * w
    f = lambda s: np.exp(1j * om * s)
    ts = dt * np.arange(1, K + 1)                      # token k sits at time (k+1) dt
    fx = f(ts)
    x = np.ones((1, K, 1, 1, 1))
    B = np.stack([fx.real, fx.imag], axis=-1).reshape(1, K, 1, 1, 2)
    C = np.zeros_like(B)
    C[..., 0] = 1.0
    full = lambda v: np.full((1, K, 1), v)
    theta = np.full((1, K, 1, 1), w)
    h0 = np.array([s0.real, s0.imag]).reshape(1, 1, 2, 1)
    Bprev = np.array([1.0, 0.0]).reshape(1, 1, 1, 2)    # f(0) enters as the carry
    xprev = np.ones((1, 1, 1, 1))
    _, h, _, _ = oracle.scan(x, B, C, full(dt), full(a), full(lam), theta, h0=h0,
                             Bprev=Bprev, xprev=xprev)
    S_num = h[0, 0, 0, 0] + 1j * h[0, 0, 1, 0]
    S_exact = np.exp(c * T) * s0 + np.exp(c * T) * (np.exp((1j * om - c) * T) - 1.0) / (1j * om - c)
    return abs(S_num - S_exact)


def test_trapezoid_convergence_order_golden():
    rows = np.loadtxt(os.path.join(GOLDEN, "trapezoid_order.txt"), ndmin=2)
    for lam, order, lo, hi in rows:
        e1 = _ode_error(lam, 0.02)
        e2 = _ode_error(lam, 0.01)
        ratio = e1 / e2
        assert lo <= ratio <= hi, (lam, order, ratio)


# --- special cases that reduce to textbook recurrences -----------------------------

def _rotation_blocks(angles):
    """Block-diagonal matrix of 2x2 rotations [[cos, -sin], [sin, cos]]."""
    K = len(angles)
    M = np.zeros((2 * K, 2 * K))
    for k, ang in enumerate(angles):
        c, s = math.cos(ang), math.sin(ang)
        M[2 * k:2 * k + 2, 2 * k:2 * k + 2] = [[c, -s], [s, c]]
    return M


def test_lambda_one_is_exponential_euler_real_rotation_form():
    """lambda = 1: h_t = e^{dt A} Rot(dt theta) h_{t-1} + dt B_t x_t^T (Mamba-2 rule + rotation).

    The real block-rotation form of the complex Euler system (linkstar.cloud
    article, section "第二刀 / Mamba-3的解法"); with theta = 0 it is Mamba-2's
    exponential-Euler recurrence (same page, "Mamba-1和Mamba-2用的是这么个离散化公式").
    """
    rng = np.random.default_rng(1)
    (x, B, C, dt, A, lam, theta), kw = rand_problem(rng, carry=True)
    lam = np.ones_like(lam)
    for th in (np.zeros_like(theta), theta):
        y, h, _, _ = oracle.scan(x, B, C, dt, A, lam, th, **kw)
        bsz, L, H, R, P = x.shape
        for b in range(bsz):
            for hh in range(H):
                S = kw["h0"][b, hh].copy()
                for t in range(L):
                    T = math.exp(dt[b, t, hh] * A[b, t, hh]) * _rotation_blocks(dt[b, t, hh] * th[b, t, hh])
                    S = T @ S + dt[b, t, hh] * (B[b, t, hh].T @ x[b, t, hh])   # (N x R)(R x P)
                    np.testing.assert_allclose(y[b, t, hh], C[b, t, hh] @ S, rtol=1e-10, atol=1e-10)
                np.testing.assert_allclose(h[b, hh], S, rtol=1e-10, atol=1e-10)


def test_theta_zero_is_real_trapezoid_ssm():
    """theta = 0: a real N-dim SSM with alpha, beta, gamma of the exponential-trapezoid rule."""
    rng = np.random.default_rng(2)
    (x, B, C, dt, A, lam, theta), kw = rand_problem(rng, carry=True)
    y, h, Bo, xo = oracle.scan(x, B, C, dt, A, lam, np.zeros_like(theta), **kw)
    bsz, L, H, R, P = x.shape
    for b in range(bsz):
        for hh in range(H):
            S = kw["h0"][b, hh].copy()
            Bp, xp = kw["Bprev"][b, hh], kw["xprev"][b, hh]
            for t in range(L):
                al = math.exp(dt[b, t, hh] * A[b, t, hh])
                be = (1 - lam[b, t, hh]) * dt[b, t, hh] * al
                ga = lam[b, t, hh] * dt[b, t, hh]
                S = al * S + be * (Bp.T @ xp) + ga * (B[b, t, hh].T @ x[b, t, hh])
                Bp, xp = B[b, t, hh], x[b, t, hh]
                np.testing.assert_allclose(y[b, t, hh], C[b, t, hh] @ S, rtol=1e-10, atol=1e-10)
            np.testing.assert_allclose(h[b, hh], S, rtol=1e-10, atol=1e-10)
            np.testing.assert_array_equal(Bo[b, hh], Bp)
            np.testing.assert_array_equal(xo[b, hh], xp)


# --- other formulations -------------------------------------------------------------

def test_complex_equals_rotated_real_rope_form():
    """The complex recurrence equals the real one with B, C rotated by the
    cumulative angle (data-dependent RoPE; linkstar.cloud article, section "RoPE技巧")."""
    rng = np.random.default_rng(3)
    (x, B, C, dt, A, lam, theta), kw = rand_problem(rng, b=2, L=17, R=3, P=4, N=8)
    y, h, _, _ = oracle.scan(x, B, C, dt, A, lam, theta, **kw)
    bsz, L, H, R, P = x.shape
    for b in range(bsz):
        for hh in range(H):
            Phi = np.cumsum(dt[b, :, hh, None] * theta[b, :, hh], axis=0)
            Bb = rot(B[b, :, hh], np.cos(Phi)[:, None], -np.sin(Phi)[:, None])
            Cb = rot(C[b, :, hh], np.cos(Phi)[:, None], -np.sin(Phi)[:, None])
            Ht = kw["h0"][b, hh].copy()
            prev = kw["Bprev"][b, hh].T @ kw["xprev"][b, hh]      # angle 0 before token 0
            for t in range(L):
                al = math.exp(dt[b, t, hh] * A[b, t, hh])
                Ht = al * (Ht + (1 - lam[b, t, hh]) * dt[b, t, hh] * prev) + \
                    lam[b, t, hh] * dt[b, t, hh] * (Bb[t].T @ x[b, t, hh])
                prev = Bb[t].T @ x[b, t, hh]
                np.testing.assert_allclose(y[b, t, hh], Cb[t] @ Ht, rtol=1e-9, atol=1e-9)
            hf = rot(Ht.T, np.cos(Phi[-1]), np.sin(Phi[-1])).T
            np.testing.assert_allclose(h[b, hh], hf, rtol=1e-9, atol=1e-9)


def test_matrix_form_semiseparable_times_two_band():
    """y = (L o C~ B~^T) X + initial-state term with L = (1-semiseparable decay) @ (2-band),
    both built as explicit dense matrices (linkstar.cloud article, section "第一刀",
    parallel form); C~, B~ are C, B rotated by the cumulative angle ("RoPE技巧")."""
    rng = np.random.default_rng(4)
    (x, B, C, dt, A, lam, theta), kw = rand_problem(rng, b=1, L=11, H=2, R=2, P=3, N=4)
    y, _, _, _ = oracle.scan(x, B, C, dt, A, lam, theta, **kw)
    _, L, H, R, P = x.shape
    for hh in range(H):
        d, a_, l_ = dt[0, :, hh], A[0, :, hh], lam[0, :, hh]
        al = np.exp(d * a_)
        # 1-semiseparable: SS[t, s] = prod_{s < u <= t} alpha_u  (t, s = 0..L-1)
        SS = np.zeros((L, L))
        for t in range(L):
            for s in range(t + 1):
                SS[t, s] = np.prod(al[s + 1:t + 1])
        # 2-band: input of step s = beta_s v_{s-1} + gamma_s v_s, v_j = B~_j x_j^T.
        # Columns are j + 1 for j = -1 .. L-1 (column 0 is the carry token j = -1).
        D2 = np.zeros((L, L + 1))
        for s in range(L):
            D2[s, s + 1] = l_[s] * d[s]
            D2[s, s] = (1 - l_[s]) * d[s] * al[s]
        Lmat = SS @ D2
        Phi = np.cumsum(d[:, None] * theta[0, :, hh], axis=0)
        Phi_full = np.concatenate([np.zeros((1, Phi.shape[1])), Phi])   # angle 0 at the carry token
        B_full = np.concatenate([kw["Bprev"][0, hh][None], B[0, :, hh]])
        X_full = np.concatenate([kw["xprev"][0, hh][None], x[0, :, hh]])
        Bt = rot(B_full, np.cos(Phi_full)[:, None], -np.sin(Phi_full)[:, None])
        Ct = rot(C[0, :, hh], np.cos(Phi)[:, None], -np.sin(Phi)[:, None])
        G = np.einsum("trn,jqn->trjq", Ct, Bt) * Lmat[:, None, :, None]
        decay0 = np.array([np.prod(al[:t + 1]) for t in range(L)])
        yy = np.einsum("trjq,jqp->trp", G, X_full) + \
            np.einsum("t,trn,np->trp", decay0, Ct, kw["h0"][0, hh])
        np.testing.assert_allclose(y[0, :, hh], yy, rtol=1e-9, atol=1e-9)


@pytest.mark.parametrize("Q", [1, 2, 3, 4, 5, 7, 8, 13, 24, 64])
def test_chunked_equals_sequential(Q):
    """The chunked decomposition (any chunk length, ragged last chunk) equals the sequential oracle."""
    rng = np.random.default_rng(5)
    (x, B, C, dt, A, lam, theta), kw = rand_problem(rng, b=2, L=24, H=2, R=2, P=3, N=6)
    y, h, _, _ = oracle.scan(x, B, C, dt, A, lam, theta, **kw)
    yc, hc = scan_chunked(x, B, C, dt, A, lam, theta, Q=Q, **kw)
    assert rel(yc, y) < 1e-12 and rel(hc, h) < 1e-12


# --- invariants ---------------------------------------------------------------------

def test_impulse_response_closed_form():
    """A single nonzero input x_s reaches y_t (t > s) with weight
    (lambda_s dt_s + (1-lambda_{s+1}) dt_{s+1}) * prod_{s<u<=t} e^{dt_u A_u} * C_t^T Rot(Phi_t - Phi_s) B_s x_s,
    and y_s = lambda_s dt_s C_s^T B_s x_s."""
    rng = np.random.default_rng(6)
    (x, B, C, dt, A, lam, theta), _ = rand_problem(rng, b=1, L=9, H=1, R=1, P=2, N=4)
    s = 3
    x = np.zeros_like(x)
    x[0, s, 0] = rng.standard_normal(x.shape[-2:])
    y, _, _, _ = oracle.scan(x, B, C, dt, A, lam, theta)
    d, a_, l_ = dt[0, :, 0], A[0, :, 0], lam[0, :, 0]
    Phi = np.cumsum(d[:, None] * theta[0, :, 0], axis=0)
    v = B[0, s, 0].T @ x[0, s, 0]                                   # N x P
    for t in range(9):
        if t < s:
            expect = np.zeros_like(y[0, t, 0])
        elif t == s:
            expect = l_[s] * d[s] * (C[0, t, 0] @ v)
        else:
            wgt = (l_[s] * d[s] + (1 - l_[s + 1]) * d[s + 1]) * np.exp(np.sum(d[s + 1:t + 1] * a_[s + 1:t + 1]))
            expect = wgt * (C[0, t, 0] @ (_rotation_blocks(Phi[t] - Phi[s]) @ v))
        np.testing.assert_allclose(y[0, t, 0], expect, rtol=1e-10, atol=1e-12)


def test_global_rotation_invariance_pins_pairing():
    """Turning every (2k, 2k+1) pair of B, C, h0 and the carry by one fixed angle leaves y
    unchanged and turns the final state by that angle (rotations of a plane commute)."""
    rng = np.random.default_rng(7)
    (x, B, C, dt, A, lam, theta), kw = rand_problem(rng, b=1, L=10, R=2, P=3, N=8)
    y, h, _, _ = oracle.scan(x, B, C, dt, A, lam, theta, **kw)
    psi = rng.uniform(-math.pi, math.pi, theta.shape[-1])
    c, s = np.cos(psi), np.sin(psi)
    kw2 = dict(kw)
    kw2["h0"] = rot(kw["h0"].swapaxes(-1, -2), c, s).swapaxes(-1, -2)
    kw2["Bprev"] = rot(kw["Bprev"], c, s)
    y2, h2, _, _ = oracle.scan(x, rot(B, c, s), rot(C, c, s), dt, A, lam, theta, **kw2)
    np.testing.assert_allclose(y2, y, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(h2, rot(h.swapaxes(-1, -2), c, s).swapaxes(-1, -2), rtol=1e-10, atol=1e-10)


def test_mimo_rank_superposition_and_rank_one():
    """The state is the sum over ranks of B_r x_r^T contributions: a rank-R run equals the
    sum of runs with one rank's x kept; and a rank-R run whose R ranks repeat one
    (B, x) pair equals the rank-1 run with x scaled by R."""
    rng = np.random.default_rng(8)
    (x, B, C, dt, A, lam, theta), kw = rand_problem(rng, b=1, L=9, R=3, P=2, N=4, h0=False, carry=False)
    y, h, _, _ = oracle.scan(x, B, C, dt, A, lam, theta)
    ys, hs = np.zeros_like(y), np.zeros_like(h)
    for r in range(3):
        xr = np.zeros_like(x)
        xr[..., r, :] = x[..., r, :]
        yr, hr, _, _ = oracle.scan(xr, B, C, dt, A, lam, theta)
        ys += yr
        hs += hr
    np.testing.assert_allclose(ys, y, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(hs, h, rtol=1e-10, atol=1e-10)
    # repeated rank
    x1, B1, C1 = x[..., :1, :], B[..., :1, :], C[..., :1, :]
    y1, h1, _, _ = oracle.scan(3 * x1, B1, C1, dt, A, lam, theta)
    yR, hR, _, _ = oracle.scan(np.repeat(x1, 3, axis=-2), np.repeat(B1, 3, axis=-2),
                               np.repeat(C1, 3, axis=-2), dt, A, lam, theta)
    np.testing.assert_allclose(hR, h1, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(yR, np.repeat(y1, 3, axis=-2), rtol=1e-10, atol=1e-10)


def test_mimo_no_cross_rank_terms():
    """B_t x_t^T pairs rank r of B with rank r of x only: moving x's rank r to rank r'
    (x_r' = x_r, x_r = 0) must change the result unless B_r = B_r'."""
    rng = np.random.default_rng(9)
    (x, B, C, dt, A, lam, theta), _ = rand_problem(rng, b=1, L=5, H=1, R=2, P=2, N=4, h0=False, carry=False)
    x[..., 1, :] = 0.0
    _, h, _, _ = oracle.scan(x, B, C, dt, A, lam, theta)
    x2 = np.zeros_like(x)
    x2[..., 1, :] = x[..., 0, :]
    B2 = B.copy()
    B2[..., 1, :] = B[..., 0, :]          # same B on the moved rank: same state
    _, h2, _, _ = oracle.scan(x2, B2, C, dt, A, lam, theta)
    np.testing.assert_allclose(h2, h, rtol=1e-12, atol=1e-12)
    _, h3, _, _ = oracle.scan(x2, B, C, dt, A, lam, theta)   # other B: different state
    assert np.max(np.abs(h3 - h)) > 1e-3


def test_linearity_in_inputs_and_initial_state():
    rng = np.random.default_rng(10)
    (x, B, C, dt, A, lam, theta), kw = rand_problem(rng)
    (x2, *_), kw2 = rand_problem(np.random.default_rng(11))
    kw2 = {"h0": kw2["h0"], "Bprev": kw["Bprev"], "xprev": kw2["xprev"]}
    y1, h1, _, _ = oracle.scan(x, B, C, dt, A, lam, theta, **kw)
    y2, h2, _, _ = oracle.scan(x2, B, C, dt, A, lam, theta, **kw2)
    kw3 = {"h0": 2 * kw["h0"] - kw2["h0"], "Bprev": kw["Bprev"], "xprev": 2 * kw["xprev"] - kw2["xprev"]}
    y3, h3, _, _ = oracle.scan(2 * x - x2, B, C, dt, A, lam, theta, **kw3)
    np.testing.assert_allclose(y3, 2 * y1 - y2, rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(h3, 2 * h1 - h2, rtol=1e-9, atol=1e-9)


def test_split_scan_with_state_and_carry_equals_full_scan():
    """Checkpoint/resume: scanning L tokens equals scanning L1 tokens, then the rest from the
    returned state and carry, and equals L - k tokens followed by k single-token steps."""
    rng = np.random.default_rng(12)
    (x, B, C, dt, A, lam, theta), kw = rand_problem(rng, b=2, L=14)
    args = (x, B, C, dt, A, lam, theta)
    y, h, Bo, xo = oracle.scan(*args, **kw)
    L1 = 6
    ya, ha, Ba, xa = oracle.scan(*(a[:, :L1] for a in args), **kw)
    yb, hb, Bb_, xb = oracle.scan(*(a[:, L1:] for a in args), h0=ha, Bprev=Ba, xprev=xa)
    np.testing.assert_allclose(np.concatenate([ya, yb], axis=1), y, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(hb, h, rtol=1e-10, atol=1e-10)
    np.testing.assert_array_equal(Bb_, Bo)
    np.testing.assert_array_equal(xb, xo)
    hs, Bs, xs = kw["h0"], kw["Bprev"], kw["xprev"]
    for t in range(14):
        yt, hs, Bs, xs = oracle.decode_step(*(a[:, t] for a in args), hs, Bs, xs)
        np.testing.assert_allclose(yt, y[:, t], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(hs, h, rtol=1e-10, atol=1e-10)


def test_zero_length_passes_state_through():
    rng = np.random.default_rng(13)
    (x, B, C, dt, A, lam, theta), kw = rand_problem(rng, L=0)
    y, h, Bo, xo = oracle.scan(x, B, C, dt, A, lam, theta, **kw)
    assert y.shape[1] == 0
    np.testing.assert_array_equal(h, kw["h0"])
    np.testing.assert_array_equal(Bo, kw["Bprev"])
    np.testing.assert_array_equal(xo, kw["xprev"])


def test_threads_do_not_change_the_result():
    rng = np.random.default_rng(14)
    (x, B, C, dt, A, lam, theta), kw = rand_problem(rng, b=3, H=5)
    r1 = oracle.scan(x, B, C, dt, A, lam, theta, nthreads=1, **kw)
    r4 = oracle.scan(x, B, C, dt, A, lam, theta, nthreads=4, **kw)
    for a, b in zip(r1, r4):
        np.testing.assert_array_equal(a, b)
