"""CPU oracle for the Mamba-3 layer recurrence -- test infrastructure only.

This package wraps ``oracle.c``: a plain sequential fp64 implementation of the
complex-valued exponential-trapezoidal recurrence with MIMO rank R (see the
header of ``oracle.c`` for the passages it follows and the readings it takes).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package.  The product library
(``selective_state_space_134_b300``) never imports it and has no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (plain C11, -O2)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", _LIB, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        d = ctypes.POINTER(ctypes.c_double)
        lib.oracle_scan.argtypes = [ctypes.c_int] * 6 + [d] * 7 + [d] * 3 + [d] * 4 + [ctypes.c_int]
        lib.oracle_scan.restype = ctypes.c_int
        lib.oracle_bc_prep.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, d, d, d,
                                       ctypes.c_double, d]
        lib.oracle_bc_prep.restype = ctypes.c_int
        lib.oracle_scan_bwd.argtypes = [ctypes.c_int] * 6 + [d] * 7 + [d] * 3 + [d] * 4 + [d] * 10
        lib.oracle_scan_bwd.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def scan(x, B, C, dt, A, lam, theta, h0=None, Bprev=None, xprev=None, nthreads: int = 1):
    """Runs the recurrence over every (b, h) sequence.

    Shapes: x [b,L,H,R,P]; B, C [b,L,H,R,N]; dt, A, lam [b,L,H]; theta [b,L,H,N/2];
    h0 [b,H,N,P] or None; Bprev [b,H,R,N] and xprev [b,H,R,P] or None.
    Returns (y [b,L,H,R,P], h_out [b,H,N,P], Bprev_out [b,H,R,N], xprev_out [b,H,R,P]),
    all float64.  With L == 0 the state and carry pass through unchanged.
    """
    x, B, C, dt, A, lam, theta = (_f64(v) for v in (x, B, C, dt, A, lam, theta))
    h0, Bprev, xprev = _f64(h0), _f64(Bprev), _f64(xprev)
    b, L, H, R, P = x.shape
    N = B.shape[-1]
    assert B.shape == (b, L, H, R, N) and C.shape == B.shape
    assert dt.shape == (b, L, H) and A.shape == dt.shape and lam.shape == dt.shape
    assert theta.shape == (b, L, H, N // 2)
    if (Bprev is None) != (xprev is None):
        raise ValueError("Bprev and xprev come together")
    y = np.zeros((b, L, H, R, P))
    h_out = np.zeros((b, H, N, P))
    Bo = np.zeros((b, H, R, N))
    xo = np.zeros((b, H, R, P))
    if L == 0:   # nothing to scan: state and carry pass through
        if h0 is not None:
            h_out[...] = h0
        if Bprev is not None:
            Bo[...] = Bprev
            xo[...] = xprev
        return y, h_out, Bo, xo
    rc = _load().oracle_scan(b, L, H, P, N, R, _ptr(x), _ptr(B), _ptr(C), _ptr(dt), _ptr(A),
                             _ptr(lam), _ptr(theta), _ptr(h0), _ptr(Bprev), _ptr(xprev),
                             _ptr(y), _ptr(h_out), _ptr(Bo), _ptr(xo), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_scan failed")
    return y, h_out, Bo, xo


def decode_step(x, B, C, dt, A, lam, theta, h, Bprev, xprev):
    """One token per (b, h): the recurrence with L = 1 (inputs without the L axis).

    Shapes: x [b,H,R,P]; B, C [b,H,R,N]; dt, A, lam [b,H]; theta [b,H,N/2];
    h [b,H,N,P]; Bprev [b,H,R,N]; xprev [b,H,R,P].
    Returns (y [b,H,R,P], h_new, Bprev_new, xprev_new).
    """
    expand = lambda a: _f64(a)[:, None]
    y, h1, Bo, xo = scan(expand(x), expand(B), expand(C), expand(dt), expand(A), expand(lam),
                         expand(theta), h0=h, Bprev=Bprev, xprev=xprev)
    return y[:, 0], h1, Bo, xo


def bc_prep(v, weight=None, bias=None, eps=1e-6):
    """BC normalisation and bias of B or C (see oracle_bc_prep in oracle.c): every row of N entries
    (one token, head and rank) becomes v / sqrt(mean(v^2) + eps) * weight[h] + bias[h, r].

    v [..., H, R, N]; weight [H, N] or None (1); bias [H, R, N] or None (0).  Returns float64.
    """
    v = _f64(v)
    H, R, N = v.shape[-3:]
    weight, bias = _f64(weight), _f64(bias)
    if weight is not None:
        assert weight.shape == (H, N)
    if bias is not None:
        assert bias.shape == (H, R, N)
    out = np.empty_like(v)
    rows = v.size // N
    if rows and _load().oracle_bc_prep(rows, H, R, N, _ptr(v), _ptr(weight), _ptr(bias), float(eps),
                                       _ptr(out)) != 0:
        raise RuntimeError("oracle_bc_prep failed")
    return out


def scan_bc(x, B, C, dt, A, lam, theta, bc, h0=None, Bprev=None, xprev=None, nthreads: int = 1):
    """The recurrence with BC normalisation and bias in front of it.

    ``bc`` = dict(B_weight, B_bias, C_weight, C_bias, eps) (None entries: 1 / 0).  B and C of every
    token, and the carry's B_prev when one is passed, go through bc_prep before the recurrence; the
    carry returned holds the raw (unnormalised) B of the last token, as the inputs gave it.
    """
    eps = bc.get("eps", 1e-6)
    Bn = bc_prep(B, bc.get("B_weight"), bc.get("B_bias"), eps)
    Cn = bc_prep(C, bc.get("C_weight"), bc.get("C_bias"), eps)
    Bpn = bc_prep(Bprev, bc.get("B_weight"), bc.get("B_bias"), eps) if Bprev is not None else None
    y, h, _, xo = scan(x, Bn, Cn, dt, A, lam, theta, h0=h0, Bprev=Bpn, xprev=xprev, nthreads=nthreads)
    L = _f64(x).shape[1]
    if L > 0:
        Bo = _f64(B)[:, -1].copy()
    else:
        Bo = _f64(Bprev).copy() if Bprev is not None else np.zeros_like(_f64(B)[:, 0])
    return y, h, Bo, xo


def decode_step_bc(x, B, C, dt, A, lam, theta, h, Bprev, xprev, bc):
    """One token per (b, h) with BC normalisation and bias (scan_bc with L = 1)."""
    expand = lambda a: _f64(a)[:, None]
    y, h1, Bo, xo = scan_bc(expand(x), expand(B), expand(C), expand(dt), expand(A), expand(lam),
                            expand(theta), bc, h0=h, Bprev=Bprev, xprev=xprev)
    return y[:, 0], h1, Bo, xo


GRAD_KEYS = ("x", "B", "C", "dt", "A", "lam", "theta")


def scan_bwd(x, B, C, dt, A, lam, theta, dy, h0=None, Bprev=None, xprev=None, dh_out=None, dBprev_out=None,
             dxprev_out=None):
    """Reverse mode of ``scan`` (oracle_scan_bwd in oracle.c): the gradient of the scalar
    sum(dy * y) + sum(dh_out * h_out) + sum(dBprev_out * Bprev_out) + sum(dxprev_out * xprev_out)
    with respect to every input.  Returns a dict with keys x, B, C, dt, A, lam, theta, h0, Bprev,
    xprev (float64, the inputs' shapes; h0 / Bprev / xprev are returned even when the inputs were
    None, i.e. zero)."""
    x, B, C, dt, A, lam, theta, dy = (_f64(v) for v in (x, B, C, dt, A, lam, theta, dy))
    h0, Bprev, xprev = _f64(h0), _f64(Bprev), _f64(xprev)
    dh_out, dBprev_out, dxprev_out = _f64(dh_out), _f64(dBprev_out), _f64(dxprev_out)
    b, L, H, R, P = x.shape
    N = B.shape[-1]
    assert dy.shape == x.shape and L >= 1
    out = {k: np.zeros_like(v) for k, v in zip(GRAD_KEYS, (x, B, C, dt, A, lam, theta))}
    out["h0"] = np.zeros((b, H, N, P))
    out["Bprev"] = np.zeros((b, H, R, N))
    out["xprev"] = np.zeros((b, H, R, P))
    rc = _load().oracle_scan_bwd(b, L, H, P, N, R, _ptr(x), _ptr(B), _ptr(C), _ptr(dt), _ptr(A), _ptr(lam),
                                 _ptr(theta), _ptr(h0), _ptr(Bprev), _ptr(xprev), _ptr(dy), _ptr(dh_out),
                                 _ptr(dBprev_out), _ptr(dxprev_out),
                                 *(_ptr(out[k]) for k in GRAD_KEYS + ("h0", "Bprev", "xprev")))
    if rc != 0:
        raise RuntimeError("oracle_scan_bwd failed")
    return out
