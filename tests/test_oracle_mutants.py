"""The oracle pins must catch plausible mistakes.

Each case below plants one mistake in a copy of ``oracle/oracle.c`` (text
substitution, compiled to a temporary library on the CPU), swaps it in for the
real oracle, and runs every pin of ``test_oracle_pins``; at least one must
fail.  The real oracle is restored afterwards.
"""
import ctypes
import inspect
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    # the left-endpoint term loses its rotation (real alpha only)
    "beta_without_rotation": ("S[k * P + p] = z[k] * (S[k * P + p] + left * u) + right * v;",
                              "S[k * P + p] = z[k] * S[k * P + p] + cabs(z[k]) * left * u + right * v;"),
    # the left-endpoint term dropped (exponential Euler with weight lambda)
    "beta_dropped": ("(S[k * P + p] + left * u)", "(S[k * P + p])"),
    # the left-endpoint term uses the current token instead of the previous one
    "beta_uses_current_token": ("u += Bp[r * K + k] * xp[r * P + p];",
                                "u += (Bt[r * N + 2 * k] + I * Bt[r * N + 2 * k + 1]) * xt[r * P + p];"),
    # beta lacks the (1 - lambda) factor
    "beta_weight_wrong": ("const double left = (1.0 - lam) * dt;", "const double left = dt;"),
    # rotation in the wrong direction
    "rotation_sign": ("I * (dt * th[k])", "-I * (dt * th[k])"),
    # C without the minus sign on its imaginary half
    "c_sign": ("Ct[r * N + 2 * k] - I * Ct[r * N + 2 * k + 1]", "Ct[r * N + 2 * k] + I * Ct[r * N + 2 * k + 1]"),
    # pairs (k, k + N/2) instead of adjacent entries, for B only
    "pairing_half_split": ("(Bt[r * N + 2 * k] + I * Bt[r * N + 2 * k + 1]) * xt[r * P + p];",
                           "(Bt[r * N + k] + I * Bt[r * N + k + K]) * xt[r * P + p];"),
    # transposed MIMO operand: rank r of B with rank (R-1-r) of x
    "mimo_cross_rank": ("* xt[r * P + p];\n", "* xt[(R - 1 - r) * P + p];\n"),
    # decay without dt
    "decay_without_dt": ("cexp(dt * A + I", "cexp(A + I"),
    # gamma uses (1 - lambda)
    "gamma_weight_wrong": ("const double right = lam * dt;", "const double right = (1.0 - lam) * dt;"),
    # not a mistake: the same product with its factors swapped must pass every pin
    "equivalent_rewrite": ("acc += creal(ck * S[k * P + p]);", "acc += creal(S[k * P + p] * ck);"),
}
EQUIVALENT = {"equivalent_rewrite"}


def _pin_functions():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        params = inspect.signature(fn).parameters
        if "Q" in params:
            out.append((name, lambda fn=fn: [fn(Q) for Q in (1, 5, 24)]))
        else:
            out.append((name, fn))
    return out


def _build_mutant(old, new, tmp):
    src = open(SRC).read()
    assert src.count(old) >= 1, old
    path = os.path.join(tmp, "mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new, 1))
    so = os.path.join(tmp, "libmutant.so")
    subprocess.run(["gcc", "-std=c11", "-O1", "-fPIC", "-shared", "-o", so, path, "-lm", "-lpthread"],
                   check=True)
    lib = ctypes.CDLL(so)
    real = oracle._load()
    lib.oracle_scan.argtypes = real.oracle_scan.argtypes
    lib.oracle_scan.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistake(mutant):
    old, new = MUTANTS[mutant]
    real = oracle._load()
    with tempfile.TemporaryDirectory() as tmp:
        oracle._lib = _build_mutant(old, new, tmp)
        try:
            failed = []
            for name, fn in _pin_functions():
                try:
                    fn()
                except AssertionError:
                    failed.append(name)
        finally:
            oracle._lib = real
    if mutant in EQUIVALENT:
        assert not failed, failed
    else:
        assert failed, f"no pin caught mutant {mutant}"
