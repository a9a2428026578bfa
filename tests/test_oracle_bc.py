"""Pins of the oracle's BC normalisation and bias (linkstar.cloud/article/869, section
"架构上的其他改动": BC归一化 -- B and C are RMS-normalised like a QK-norm; BC偏置 -- a learnable,
data-independent bias is added to B and C).

The reading taken: every (token, head, rank) row of N entries becomes
v / sqrt(mean(v^2) + eps) * weight[h] + bias[h, r]; the carry keeps the raw B of the last token
and is normalised where it is consumed.  Each pin is fixed by something other than the oracle's own
formula: a property of the normalisation (unit RMS rows, invariance to a positive scale of a row, a
fixed point), a closed form (a constant row; the response of the recurrence to the bias alone, a
geometric series), or the split-and-resume identity of the recurrence.  The planted-mistake cases at
the end check that these pins catch the plausible errors.
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def _rand_problem(rng, b=2, L=13, H=3, R=2, P=3, N=6):
    x = rng.standard_normal((b, L, H, R, P))
    B = rng.standard_normal((b, L, H, R, N))
    C = rng.standard_normal((b, L, H, R, N))
    dt = np.log1p(np.exp(rng.standard_normal((b, L, H)) - 1.0))
    A = -np.exp(0.5 * rng.standard_normal((b, L, H)))
    lam = 1.0 / (1.0 + np.exp(-rng.standard_normal((b, L, H))))
    theta = rng.uniform(-np.pi, np.pi, (b, L, H, N // 2))
    return x, B, C, dt, A, lam, theta


def _rand_bc(rng, H, R, N, eps):
    return dict(B_weight=rng.uniform(0.5, 1.5, (H, N)), B_bias=0.3 * rng.standard_normal((H, R, N)),
                C_weight=rng.uniform(0.5, 1.5, (H, N)), C_bias=0.3 * rng.standard_normal((H, R, N)), eps=eps)


def test_rows_have_unit_rms_and_the_gain_is_per_head():
    # eps = 0, zero bias: prep(v)[..., h, r, :] / weight[h] has RMS exactly 1 for every row, so the
    # statistic runs over the N entries of one (token, head, rank) row and the gain is head h's
    rng = np.random.default_rng(1)
    v = rng.standard_normal((4, 7, 3, 2, 8)) * rng.uniform(0.1, 10.0, (4, 7, 3, 2, 1))
    w = rng.uniform(0.5, 2.0, (3, 8))
    out = oracle.bc_prep(v, weight=w, eps=0.0)
    ratio = out / w[None, None, :, None, :]
    np.testing.assert_allclose(np.sqrt(np.mean(ratio ** 2, axis=-1)), 1.0, rtol=1e-13)
    # the normalised row keeps the direction of the raw row
    cos = np.sum(ratio * v, -1) / np.linalg.norm(ratio, axis=-1) / np.linalg.norm(v, axis=-1)
    np.testing.assert_allclose(cos, 1.0, rtol=1e-13)


def test_constant_row_closed_form_places_eps_inside_the_mean():
    # a row of N equal entries c with eps = 3 c^2: c / sqrt(c^2 + 3 c^2) = sign(c) / 2
    N, H, R = 8, 2, 3
    c = np.array([0.7, -2.5, 1e-3]).reshape(1, 1, 3, 1) * np.ones((1, H, R, N))
    rng = np.random.default_rng(2)
    for i in range(R):
        row = np.full((1, H, 1, N), c[0, 0, i, 0])
        eps = 3.0 * c[0, 0, i, 0] ** 2
        w = rng.uniform(0.5, 2.0, (H, N))
        bias = rng.standard_normal((H, 1, N))
        out = oracle.bc_prep(row, weight=w, bias=bias, eps=eps)
        want = 0.5 * np.sign(c[0, 0, i, 0]) * w[:, None, :] + bias
        np.testing.assert_allclose(out[0], want, rtol=1e-13, atol=1e-15)


def test_unit_rms_rows_are_a_fixed_point():
    # unit gain, zero bias, eps = 0: rows that already have RMS 1 pass through, and the normalised
    # recurrence equals the plain one on them
    rng = np.random.default_rng(3)
    x, B, C, dt, A, lam, theta = _rand_problem(rng)
    N = B.shape[-1]
    B = B / np.sqrt(np.mean(B * B, -1, keepdims=True))
    C = C / np.sqrt(np.mean(C * C, -1, keepdims=True))
    y0, h0, _, _ = oracle.scan(x, B, C, dt, A, lam, theta)
    y1, h1, _, _ = oracle.scan_bc(x, B, C, dt, A, lam, theta, dict(eps=0.0))
    np.testing.assert_allclose(y1, y0, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(h1, h0, rtol=1e-12, atol=1e-12)
    assert N == 6


def test_output_is_invariant_to_a_positive_scale_of_each_row():
    # eps = 0: scaling every B and C row by its own positive factor changes nothing downstream
    rng = np.random.default_rng(4)
    x, B, C, dt, A, lam, theta = _rand_problem(rng)
    H, R, N = B.shape[2:]
    bc = _rand_bc(rng, H, R, N, 0.0)
    y0, h0, _, _ = oracle.scan_bc(x, B, C, dt, A, lam, theta, bc)
    sB = rng.uniform(0.01, 100.0, B.shape[:-1] + (1,))
    sC = rng.uniform(0.01, 100.0, C.shape[:-1] + (1,))
    y1, h1, _, _ = oracle.scan_bc(x, B * sB, C * sC, dt, A, lam, theta, bc)
    np.testing.assert_allclose(y1, y0, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(h1, h0, rtol=1e-10, atol=1e-10)


def test_bias_alone_gives_the_geometric_series_response():
    # B = C = 0 (eps > 0: a zero row normalises to 0), theta = 0, P = 1, x = 1, constant dt, A,
    # lambda: B'_t = bias_B[h, r], C'_t = bias_C[h, r] for every token, so with
    # alpha = e^{dt A}, beta = (1 - lambda) dt alpha, gamma = lambda dt:
    #   h_t = alpha^t gamma u + (beta + gamma) u (1 - alpha^t) / (1 - alpha),  u = sum_r bias_B[h, r]
    #   y_t[r] = <bias_C[h, r], h_t>
    rng = np.random.default_rng(5)
    b, L, H, R, N = 1, 40, 3, 2, 4
    dtv, Av, lv = 0.3, -0.8, 0.35
    x = np.ones((b, L, H, R, 1))
    B = np.zeros((b, L, H, R, N))
    C = np.zeros((b, L, H, R, N))
    dt = np.full((b, L, H), dtv)
    A = np.full((b, L, H), Av)
    lam = np.full((b, L, H), lv)
    theta = np.zeros((b, L, H, N // 2))
    bc = dict(B_weight=rng.uniform(0.5, 2.0, (H, N)), B_bias=rng.standard_normal((H, R, N)),
              C_weight=rng.uniform(0.5, 2.0, (H, N)), C_bias=rng.standard_normal((H, R, N)), eps=1e-6)
    y, h, _, _ = oracle.scan_bc(x, B, C, dt, A, lam, theta, bc)
    alpha = np.exp(dtv * Av)
    beta, gamma = (1 - lv) * dtv * alpha, lv * dtv
    t = np.arange(L)
    coef = alpha ** t * gamma + (beta + gamma) * (1 - alpha ** t) / (1 - alpha)
    for hh in range(H):
        u = bc["B_bias"][hh].sum(0)                         # [N]
        for r in range(R):
            want = coef * (bc["C_bias"][hh, r] @ u)
            np.testing.assert_allclose(y[0, :, hh, r, 0], want, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(h[0, hh, :, 0], coef[-1] * u, rtol=1e-12)


def test_split_scan_with_raw_carry_equals_the_whole_scan():
    # the carry returned holds the raw B of the last token; resuming from it (the next call
    # normalises it where it is consumed) reproduces the single long scan
    rng = np.random.default_rng(6)
    x, B, C, dt, A, lam, theta = _rand_problem(rng, L=17)
    H, R, N = B.shape[2:]
    bc = _rand_bc(rng, H, R, N, 0.25)
    y, h, Bo, xo = oracle.scan_bc(x, B, C, dt, A, lam, theta, bc)
    np.testing.assert_array_equal(Bo, B[:, -1])
    for L1 in (1, 6, 16):
        a = [v[:, :L1] for v in (x, B, C, dt, A, lam, theta)]
        c = [v[:, L1:] for v in (x, B, C, dt, A, lam, theta)]
        y1, h1, B1, x1 = oracle.scan_bc(*a, bc)
        y2, h2, B2, x2 = oracle.scan_bc(*c, bc, h0=h1, Bprev=B1, xprev=x1)
        np.testing.assert_allclose(np.concatenate([y1, y2], 1), y, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(h2, h, rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(B2, Bo)
    # and token by token through the decode step
    st = (np.zeros_like(h), np.zeros_like(Bo), np.zeros_like(xo))
    ys = []
    for t in range(x.shape[1]):
        yt, *st = oracle.decode_step_bc(*(v[:, t] for v in (x, B, C, dt, A, lam, theta)), *st, bc)
        ys.append(yt)
    np.testing.assert_allclose(np.stack(ys, 1), y, rtol=1e-12, atol=1e-12)


def _bc_pins():
    return [fn for name, fn in sorted(globals().items())
            if name.startswith("test_") and callable(fn) and name not in ("test_bc_pins_catch_planted_mistake",
                                                                            "test_carry_mistake_is_caught")]


BC_MUTANTS = {
    # the mean square over the wrong count (the sum of squares, not the mean)
    "sum_not_mean": ("        ms /= N;\n", ""),
    # eps added outside the square root
    "eps_outside_sqrt": ("1.0 / sqrt(ms + eps)", "1.0 / (sqrt(ms) + eps)"),
    # no square root (divides by the mean square)
    "no_sqrt": ("1.0 / sqrt(ms + eps)", "1.0 / (ms + eps)"),
    # bias added before the normalisation
    "bias_before_norm": ("o[n] = row[n] * inv * g + c;", "o[n] = (row[n] + c) * inv * g;"),
    # the gain of head 0 for every head
    "gain_head_zero": ("weight[(size_t)h * N + n]", "weight[n]"),
    # the bias of rank 0 for every rank
    "bias_rank_zero": ("bias[((size_t)h * R + r) * N + n]", "bias[((size_t)h * R) * N + n]"),
    # not a mistake: the same product regrouped must pass every pin
    "equivalent_rewrite": ("o[n] = row[n] * inv * g + c;", "o[n] = c + g * (row[n] * inv);"),
}


def _build_mutant(old, new, tmp):
    src = open(SRC).read()
    assert src.count(old) == 1, old
    path = os.path.join(tmp, "mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new, 1))
    so = os.path.join(tmp, "libmutant.so")
    subprocess.run(["gcc", "-std=c11", "-O1", "-fPIC", "-shared", "-o", so, path, "-lm", "-lpthread"], check=True)
    lib = ctypes.CDLL(so)
    real = oracle._load()
    for fn in ("oracle_scan", "oracle_bc_prep"):
        getattr(lib, fn).argtypes = getattr(real, fn).argtypes
        getattr(lib, fn).restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("mutant", sorted(BC_MUTANTS))
def test_bc_pins_catch_planted_mistake(mutant):
    old, new = BC_MUTANTS[mutant]
    real = oracle._load()
    with tempfile.TemporaryDirectory() as tmp:
        oracle._lib = _build_mutant(old, new, tmp)
        try:
            failed = []
            for fn in _bc_pins():
                try:
                    fn()
                except AssertionError:
                    failed.append(fn.__name__)
        finally:
            oracle._lib = real
    if mutant == "equivalent_rewrite":
        assert not failed, failed
    else:
        assert failed, f"no pin caught mutant {mutant}"


def test_carry_mistake_is_caught(monkeypatch):
    # a carry that holds the normalised B (and is normalised again where it is consumed) breaks the
    # split-and-resume pin
    real = oracle.scan_bc

    def wrong(x, B, C, dt, A, lam, theta, bc, h0=None, Bprev=None, xprev=None, nthreads=1):
        y, h, Bo, xo = real(x, B, C, dt, A, lam, theta, bc, h0=h0, Bprev=Bprev, xprev=xprev, nthreads=nthreads)
        return y, h, oracle.bc_prep(Bo, bc.get("B_weight"), bc.get("B_bias"), bc.get("eps", 1e-6)), xo

    monkeypatch.setattr(oracle, "scan_bc", wrong)
    with pytest.raises(AssertionError):
        test_split_scan_with_raw_carry_equals_the_whole_scan()
