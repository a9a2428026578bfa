"""GPU parity of the BC normalisation and bias (linkstar.cloud/article/869, section
"架构上的其他改动": BC归一化, BC偏置) fused into the prefill and decode kernels, against the fp64 oracle
(oracle.scan_bc / oracle.decode_step_bc) on the same seeded inputs and synthetic gains and biases.

Tolerances as for the plain recurrence: max|y - y_ref| / rms(y_ref) <= 2e-2 for bf16 inputs on the
tensor-core path, 1e-4 for fp32 inputs; the carry returned is the raw B of the last token.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_134_b300 as m3
from selective_state_space_134_b300.synth import WORKLOADS, bc_params, decode_pool, decode_state, prefill_inputs, to_f64
from helpers import KEYS, TOL, assert_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_134_b300 import build
    build.build()
    torch.cuda.init()


def _bc(w, seed=0, eps=1e-5, drop=()):
    p = bc_params(w, "cuda", seed=seed, eps=eps)
    for k in drop:
        p[k] = None
    dev = m3.BcNorm(p["B_weight"], p["B_bias"], p["C_weight"], p["C_bias"], eps)
    ref = {k: (to_f64(v) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
    return dev, ref


def _state(w, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return m3.State(torch.randn(w.batch, w.nheads, w.N, w.P, device="cuda", generator=g),
                    (2.0 * torch.randn(w.batch, w.nheads, w.R, w.N, device="cuda", generator=g)).to(dtype),
                    torch.randn(w.batch, w.nheads, w.R, w.P, device="cuda", generator=g).to(dtype))


CASES = {
    # tensor-core path (bf16, P = 64)
    "siso_n64": ("siso_n64", dict(batch=2, nheads=3, seqlen=300)),
    "siso_n128": ("siso_n128", dict(batch=1, nheads=2, seqlen=333)),
    "mimo_r4": ("mimo_r4", dict(batch=1, nheads=3, seqlen=201)),
    "mimo_r8_n128": ("mimo_r4", dict(batch=1, nheads=2, seqlen=150, R=8, N=128)),
    "long_segmented": ("long_n128_r4", dict(batch=1, nheads=2, seqlen=1100)),
    # SIMT path (fp32 inputs, other shapes), one case segmented
    "tiny_f32": ("tiny_f32", {}),
    "siso_f32": ("siso_n64", dict(batch=1, nheads=2, seqlen=300, dtype="f32")),
    "mimo_f32_segmented": ("mimo_r4", dict(batch=1, nheads=1, seqlen=777, dtype="f32")),
    "odd_bf16": ("tiny_f32", dict(N=6, P=8, R=2, seqlen=65, nheads=2, dtype="bf16")),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("with_state", [False, True])
def test_prefill_bc_matches_oracle(case, with_state):
    wname, over = CASES[case]
    w = WORKLOADS[wname].with_(**over)
    inp = prefill_inputs(w, "cuda")
    bc, bref = _bc(w, seed=1)
    st = _state(w, inp["x"].dtype, 5) if with_state else None
    so = m3.State.zeros(w.batch, w.nheads, w.P, w.N, w.R, inp["x"].dtype)
    y = m3.scan_fwd(*(inp[k] for k in KEYS), state_in=st, state_out=so, bc=bc)
    assert m3.device_status() == m3.M3_OK
    kw = {}
    if st is not None:
        kw = dict(h0=to_f64(st.h), Bprev=to_f64(st.B_prev), xprev=to_f64(st.x_prev))
    yr, hr, Br, xr = oracle.scan_bc(*(to_f64(inp[k]) for k in KEYS), bref, nthreads=8, **kw)
    tol = TOL[w.dtype]
    assert_err(to_f64(y), yr, tol, "y")
    assert_err(to_f64(so.h), hr, tol, "h")
    np.testing.assert_array_equal(to_f64(so.B_prev), Br)      # the raw B of the last token
    np.testing.assert_array_equal(to_f64(so.x_prev), xr)


@pytest.mark.parametrize("drop", [("B_weight", "C_weight"), ("B_bias", "C_bias"), ("B_weight", "B_bias")])
def test_prefill_bc_optional_gain_and_bias(drop):
    # NULL gain = 1, NULL bias = 0, independently for B and C
    w = WORKLOADS["mimo_r4"].with_(batch=1, nheads=2, seqlen=180)
    inp = prefill_inputs(w, "cuda")
    bc, bref = _bc(w, seed=2, drop=drop)
    y = m3.scan_fwd(*(inp[k] for k in KEYS), bc=bc)
    yr, _, _, _ = oracle.scan_bc(*(to_f64(inp[k]) for k in KEYS), bref)
    assert_err(to_f64(y), yr, TOL[w.dtype], "y")


@pytest.mark.parametrize("wname", ["siso_n64", "mimo_r4"])
def test_prefill_bc_full_size_sampled(wname):
    w = WORKLOADS[wname]
    inp = prefill_inputs(w, "cuda")
    bc, bref = _bc(w, seed=3)
    so = m3.State.zeros(w.batch, w.nheads, w.P, w.N, w.R, inp["x"].dtype)
    y = m3.scan_fwd(*(inp[k] for k in KEYS), state_out=so, bc=bc)
    assert m3.device_status() == m3.M3_OK
    pairs = [(0, 0), (w.batch - 1, w.nheads - 1)]
    for b, h in pairs:
        one = {k: to_f64(inp[k][b:b + 1, :, h:h + 1]) for k in KEYS}
        ref1 = {k: (v[h:h + 1] if isinstance(v, np.ndarray) else v) for k, v in bref.items()}
        yr, hr, _, _ = oracle.scan_bc(*(one[k] for k in KEYS), ref1)
        assert_err(to_f64(y[b:b + 1, :, h:h + 1]), yr, TOL[w.dtype], f"y {(b, h)}")
        assert_err(to_f64(so.h[b:b + 1, h:h + 1]), hr, TOL[w.dtype], f"h {(b, h)}")


@pytest.mark.parametrize("over,variant", [(dict(), m3.DECODE_STREAM), (dict(N=128, R=4), m3.DECODE_STREAM),
                                          (dict(dtype="f32"), m3.DECODE_STREAM),
                                          (dict(P=16, dtype="f32", R=2), m3.DECODE_GENERIC),
                                          (dict(P=16, N=6, R=3), m3.DECODE_GENERIC)])
def test_decode_bc_matches_oracle(over, variant):
    # BC-normalised decode runs on the per-thread FMA kernels (streaming or generic)
    w = WORKLOADS["decode_n64_r4"].with_(batch=3, nheads=7, **over)
    st = decode_state(w, "cuda")
    state = m3.State(st["h"].clone(), st["B_prev"].clone(), st["x_prev"].clone())
    bc, bref = _bc(w, seed=4)
    ref = [to_f64(st["h"]), to_f64(st["B_prev"]), to_f64(st["x_prev"])]
    for step, tok in enumerate(decode_pool(w, "cuda", pool=3)):
        y = m3.decode_step(*(tok[k] for k in KEYS), state=state, bc=bc)
        assert m3.decode_last_variant() == variant
        assert m3.device_status() == m3.M3_OK
        yr, *ref = oracle.decode_step_bc(*(to_f64(tok[k]) for k in KEYS), *ref, bref)
        assert_err(to_f64(y), yr, 1e-5, f"y {step}")
        assert_err(to_f64(state.h), ref[0], 1e-5, f"h {step}")
        np.testing.assert_array_equal(to_f64(state.B_prev), ref[1])


def test_bc_prefill_then_decode_equals_full_prefill():
    # a prefill of the first tokens, then decode steps from its state and raw carry, equals one
    # prefill over all tokens (both with BC normalisation)
    w = WORKLOADS["siso_n64"].with_(batch=2, nheads=3, seqlen=160)
    inp = prefill_inputs(w, "cuda")
    bc, _ = _bc(w, seed=6)
    y_full = m3.scan_fwd(*(inp[k] for k in KEYS), bc=bc)
    L1 = 150
    st = m3.State.zeros(w.batch, w.nheads, w.P, w.N, w.R, inp["x"].dtype)
    y1 = m3.scan_fwd(*(inp[k][:, :L1].contiguous() for k in KEYS), state_out=st, bc=bc)
    ys = [y1]
    for t in range(L1, w.seqlen):
        ys.append(m3.decode_step(*(inp[k][:, t].contiguous() for k in KEYS), state=st, bc=bc).unsqueeze(1))
    assert_err(to_f64(torch.cat(ys, 1)), to_f64(y_full), TOL[w.dtype], "y")
