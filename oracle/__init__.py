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
