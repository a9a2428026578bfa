"""Shared helpers of the tests: error metric, oracle on sampled (b, h) slices."""
import os

import numpy as np
import torch

import oracle
from selective_state_space_134_b300.synth import to_f64

TOL = {"f32": 1e-4, "bf16": 2e-2}   # max|y - y_ref| / rms(y_ref)
KEYS = ("x", "B", "C", "dt", "A", "lam", "theta")


# (test id, what, measured error, bar) of every checked comparison in this process; conftest.py
# prints the ones closest to their bar at the end of the run
RECORD = []


def norm_err(got, ref, floor=1e-30) -> float:
    """max|got - ref| / rms(ref); the denominator is at least `floor` (for references that vanish)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.max(np.abs(got - ref)) / max(rms, floor))


def assert_err(got, ref, tol, what="", floor=1e-30) -> float:
    """Asserts norm_err(got, ref, floor) <= tol and records the measured error against its bar."""
    e = norm_err(got, ref, floor)
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    RECORD.append((test, str(what), e, float(tol)))
    assert e <= tol, (what, e, tol)
    return e


def slice_inputs(inp: dict, b: int, h: int) -> dict:
    """One (b, h) sequence of prefill inputs as float64 numpy, shaped batch = 1, heads = 1."""
    out = {}
    for k in KEYS:
        t = inp[k][b:b + 1, :, h:h + 1]
        out[k] = to_f64(t)
    return out


def oracle_slices(inp: dict, pairs, state_in=None, nthreads=1):
    """Runs the oracle on the given (b, h) pairs; returns lists of (y, h_out, Bprev, xprev)."""
    res = []
    for b, h in pairs:
        s = slice_inputs(inp, b, h)
        kw = {}
        if state_in is not None:
            kw["h0"] = to_f64(state_in.h[b:b + 1, h:h + 1])
            if state_in.B_prev is not None:
                kw["Bprev"] = to_f64(state_in.B_prev[b:b + 1, h:h + 1])
                kw["xprev"] = to_f64(state_in.x_prev[b:b + 1, h:h + 1])
        res.append(oracle.scan(*(s[k] for k in KEYS), nthreads=nthreads, **kw))
    return res


def oracle_full(inp: dict, state_in=None, nthreads=8):
    kw = {}
    if state_in is not None:
        kw["h0"] = to_f64(state_in.h)
        if state_in.B_prev is not None:
            kw["Bprev"] = to_f64(state_in.B_prev)
            kw["xprev"] = to_f64(state_in.x_prev)
    return oracle.scan(*(to_f64(inp[k]) for k in KEYS), nthreads=nthreads, **kw)


def to_dev(inp: dict, device="cuda") -> dict:
    return {k: v.to(device) for k, v in inp.items()}
