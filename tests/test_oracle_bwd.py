"""Pins of the oracle's backward pass (oracle.scan_bwd, the reverse mode of the recurrence used to
train it; linkstar.cloud/article/869, section "训练怎么办").

The gradients are fixed by something other than the adjoint's own algebra: central finite
differences of the forward oracle (itself pinned by test_oracle_pins) on small problems, for every
input including the initial state and carry and with gradients flowing in through y, the final
state and the carry; and a closed-form derivative of a one-pair, one-token case.  The planted
mistakes at the end check that these pins catch plausible errors in the adjoint.
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")
IN = ("x", "B", "C", "dt", "A", "lam", "theta", "h0", "Bprev", "xprev")


def _problem(rng, b=1, L=6, H=2, R=2, P=3, N=4, carry=True):
    d = dict(x=rng.standard_normal((b, L, H, R, P)), B=rng.standard_normal((b, L, H, R, N)),
             C=rng.standard_normal((b, L, H, R, N)), dt=np.log1p(np.exp(rng.standard_normal((b, L, H)) - 1.0)),
             A=-np.exp(0.5 * rng.standard_normal((b, L, H))),
             lam=1.0 / (1.0 + np.exp(-rng.standard_normal((b, L, H)))),
             theta=rng.uniform(-np.pi, np.pi, (b, L, H, N // 2)), h0=rng.standard_normal((b, H, N, P)))
    if carry:
        d["Bprev"] = rng.standard_normal((b, H, R, N))
        d["xprev"] = rng.standard_normal((b, H, R, P))
    else:
        d["Bprev"] = d["xprev"] = None
    return d


def _loss(d, w):
    y, h, Bo, xo = oracle.scan(*(d[k] for k in oracle.GRAD_KEYS), h0=d["h0"], Bprev=d["Bprev"], xprev=d["xprev"])
    return float(np.sum(w["dy"] * y) + np.sum(w["dh"] * h) + np.sum(w["dBo"] * Bo) + np.sum(w["dxo"] * xo))


def _weights(rng, d):
    b, L, H, R, P = d["x"].shape
    N = d["B"].shape[-1]
    return dict(dy=rng.standard_normal((b, L, H, R, P)), dh=rng.standard_normal((b, H, N, P)),
                dBo=rng.standard_normal((b, H, R, N)), dxo=rng.standard_normal((b, H, R, P)))


@pytest.mark.parametrize("shape", [dict(), dict(R=1, N=2, P=1, L=5), dict(b=2, L=4, H=1, R=3, P=2, N=6),
                                   dict(carry=False, L=3)])
def test_adjoint_matches_central_differences(shape):
    rng = np.random.default_rng(11)
    d = _problem(rng, **shape)
    w = _weights(rng, d)
    g = oracle.scan_bwd(*(d[k] for k in oracle.GRAD_KEYS), w["dy"], h0=d["h0"], Bprev=d["Bprev"],
                        xprev=d["xprev"], dh_out=w["dh"], dBprev_out=w["dBo"], dxprev_out=w["dxo"])
    eps = 1e-6
    for k in IN:
        if d[k] is None:
            assert not np.any(g[k][..., :0])
            continue
        fd = np.zeros_like(d[k])
        flat, ff = d[k].reshape(-1), fd.reshape(-1)
        for i in range(flat.size):
            v = flat[i]
            flat[i] = v + eps
            lp = _loss(d, w)
            flat[i] = v - eps
            lm = _loss(d, w)
            flat[i] = v
            ff[i] = (lp - lm) / (2 * eps)
        scale = max(1.0, float(np.max(np.abs(fd))))
        np.testing.assert_allclose(g[k], fd, rtol=0, atol=2e-7 * scale, err_msg=k)


def test_one_pair_one_token_closed_form():
    # N = 2, P = R = 1, L = 1, no carry: S = z h0 + right v, y = Re(Cc S) with z = e^{dt(A + i theta)},
    # v = (B0 + i B1) x, Cc = C0 - i C1.  With dy = 1, the derivatives are those of
    #   y = C0 Re(S) + C1 Im(S),
    # e.g. dy/dA = dt Re(Cc z h0c), dy/dtheta = dt Re(Cc i z h0c), dy/dlam = dt Re(Cc v),
    # dy/dx = lam dt Re(Cc (B0 + i B1)), dy/dh0 = (Re(Cc z), -Im(Cc z)) as real / imaginary parts.
    dtv, Av, lv, th, xv = 0.7, -0.4, 0.3, 1.1, 0.9
    B0, B1, C0, C1, h0r, h0i = 0.5, -1.2, 0.8, 0.35, -0.6, 1.4
    f = lambda a: np.array(a, dtype=float).reshape
    x = np.array([xv]).reshape(1, 1, 1, 1, 1)
    B = np.array([B0, B1]).reshape(1, 1, 1, 1, 2)
    C = np.array([C0, C1]).reshape(1, 1, 1, 1, 2)
    dt, A, lam = (np.array([v]).reshape(1, 1, 1) for v in (dtv, Av, lv))
    theta = np.array([th]).reshape(1, 1, 1, 1)
    h0 = np.array([h0r, h0i]).reshape(1, 1, 2, 1)
    g = oracle.scan_bwd(x, B, C, dt, A, lam, theta, np.ones((1, 1, 1, 1, 1)), h0=h0)
    z = np.exp(dtv * (Av + 1j * th))
    hc, bc, cc = h0r + 1j * h0i, B0 + 1j * B1, C0 - 1j * C1
    v = bc * xv
    S = z * hc + lv * dtv * v
    np.testing.assert_allclose(g["A"].item(), dtv * (cc * z * hc).real, rtol=1e-13)
    np.testing.assert_allclose(g["theta"].item(), dtv * (cc * 1j * z * hc).real, rtol=1e-13)
    np.testing.assert_allclose(g["lam"].item(), dtv * (cc * v).real, rtol=1e-13)
    np.testing.assert_allclose(g["dt"].item(), ((Av + 1j * th) * cc * z * hc).real + lv * (cc * v).real, rtol=1e-13)
    np.testing.assert_allclose(g["x"].item(), lv * dtv * (cc * bc).real, rtol=1e-13)
    np.testing.assert_allclose(g["B"].ravel(), [lv * dtv * xv * C0, lv * dtv * xv * C1], rtol=1e-13)
    np.testing.assert_allclose(g["C"].ravel(), [S.real, S.imag], rtol=1e-13)
    np.testing.assert_allclose(g["h0"].ravel(), [(cc * z).real, -(cc * z).imag], rtol=1e-13)


def _pins():
    return [lambda: test_adjoint_matches_central_differences(dict()),
            lambda: test_adjoint_matches_central_differences(dict(carry=False, L=3)),
            test_one_pair_one_token_closed_form]


BWD_MUTANTS = {
    # the state gradient passes back through z instead of conj(z)
    "transition_not_conjugated": ("const double complex gw = conj(z) * g;", "const double complex gw = z * g;"),
    # the angle gradient takes the real part (the decay's) instead of the imaginary part
    "angle_real_part": ("dom += cimag(q);", "dom += creal(q);"),
    # the left-endpoint gradient uses G instead of G_W
    "left_uses_G": ("dleft += creal(conj(u) * gw);", "dleft += creal(conj(u) * g);"),
    # lambda's gradient with the wrong sign on the left term
    "lambda_sign": ("gr->dlam[tok] = dt * (dright - dleft);", "gr->dlam[tok] = dt * (dright + dleft);"),
    # C's imaginary half without its sign convention
    "c_imag_sign": ("G[k * P + p] += dyt[r * P + p] * (Ct[r * N + 2 * k] + I * Ct[r * N + 2 * k + 1]);",
                    "G[k * P + p] += dyt[r * P + p] * (Ct[r * N + 2 * k] - I * Ct[r * N + 2 * k + 1]);"),
}


@pytest.mark.parametrize("mutant", sorted(BWD_MUTANTS))
def test_bwd_pins_catch_planted_mistake(mutant):
    old, new = BWD_MUTANTS[mutant]
    real = oracle._load()
    with tempfile.TemporaryDirectory() as tmp:
        src = open(SRC).read()
        assert src.count(old) == 1, old
        path = os.path.join(tmp, "mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new, 1))
        so = os.path.join(tmp, "libmutant.so")
        subprocess.run(["gcc", "-std=c11", "-O1", "-fPIC", "-shared", "-o", so, path, "-lm", "-lpthread"], check=True)
        lib = ctypes.CDLL(so)
        for fn in ("oracle_scan", "oracle_scan_bwd", "oracle_bc_prep"):
            getattr(lib, fn).argtypes = getattr(real, fn).argtypes
            getattr(lib, fn).restype = ctypes.c_int
        oracle._lib = lib
        try:
            failed = 0
            for pin in _pins():
                try:
                    pin()
                except AssertionError:
                    failed += 1
        finally:
            oracle._lib = real
    assert failed, f"no pin caught mutant {mutant}"
