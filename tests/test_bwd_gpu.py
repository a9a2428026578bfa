"""GPU parity of the backward pass (mamba3_scan_bwd, reverse mode of the chunked recurrence for
training; linkstar.cloud/article/869, section "训练怎么办") against the oracle's sequential fp64
adjoint (oracle.scan_bwd, itself pinned by finite differences of the forward oracle).

The kernel computes in fp32 on exactly the stored inputs, so every gradient tensor is held to
max|g - g_ref| / rms(g_ref) <= 1e-4, the bar of an fp32 forward; inputs bf16 or fp32, several chunks
with a ragged tail, an initial state and carry, and gradients flowing in through y, the final state
and the carry.  A gradient that vanishes identically (theta's for one token from a zero state: the
rotation of B and C by one angle leaves the output unchanged) is held to |g| <= 1e-4 x 1e-3 in
absolute terms (the denominator floored at 1e-3; the inputs and dy are of order one).
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_134_b300 as m3
from selective_state_space_134_b300.synth import WORKLOADS, prefill_inputs, to_f64
from helpers import KEYS, assert_err

pytestmark = pytest.mark.gpu
BAR = 1e-4
GKEYS = ("x", "B", "C", "dt", "A", "lam", "theta")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_134_b300 import build
    build.build()
    torch.cuda.init()


def _rand(shape, seed, scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return scale * torch.randn(shape, device="cuda", generator=g)


CASES = {
    "tiny_f32": ("tiny_f32", dict(seqlen=100)),
    "siso_n64_bf16": ("siso_n64", dict(batch=1, nheads=2, seqlen=100)),
    "siso_n128_bf16": ("siso_n128", dict(batch=1, nheads=2, seqlen=70)),
    "mimo_r4_bf16": ("mimo_r4", dict(batch=2, nheads=1, seqlen=67)),
    "mimo_r8_f32": ("mimo_r4", dict(batch=1, nheads=1, seqlen=21, R=8, dtype="f32")),
    "odd_f32": ("tiny_f32", dict(N=6, P=8, R=3, seqlen=37, nheads=2)),
    "odd_bf16": ("tiny_f32", dict(N=6, P=8, R=3, seqlen=37, nheads=2, dtype="bf16")),
    "mimo_r8_bf16": ("mimo_r4", dict(batch=1, nheads=2, seqlen=45, R=8)),
    # fp32 N = 128: one state tile in shared memory (H'_{c+1} read back from the checkpoints)
    "siso_n128_f32": ("siso_n128", dict(batch=1, nheads=1, seqlen=40, dtype="f32")),
    "single_token": ("siso_n64", dict(batch=2, nheads=1, seqlen=1)),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("with_state", [False, True])
def test_backward_matches_oracle(case, with_state):
    wname, over = CASES[case]
    w = WORKLOADS[wname].with_(**over)
    inp = prefill_inputs(w, "cuda")
    b, H, R, P, N = w.batch, w.nheads, w.R, w.P, w.N
    dy = _rand(inp["x"].shape, 1)
    st, dh, dBo, dxo = None, None, None, None
    if with_state:
        st = m3.State(_rand((b, H, N, P), 2), _rand((b, H, R, N), 3).to(inp["x"].dtype),
                      _rand((b, H, R, P), 4).to(inp["x"].dtype))
        dh, dBo, dxo = _rand((b, H, N, P), 5), _rand((b, H, R, N), 6), _rand((b, H, R, P), 7)
    g = m3.scan_bwd(*(inp[k] for k in KEYS), dy, state_in=st, dh_out=dh, dB_prev_out=dBo, dx_prev_out=dxo)
    assert m3.device_status() == m3.M3_OK
    kw = {}
    if with_state:
        kw = dict(h0=to_f64(st.h), Bprev=to_f64(st.B_prev), xprev=to_f64(st.x_prev), dh_out=to_f64(dh),
                  dBprev_out=to_f64(dBo), dxprev_out=to_f64(dxo))
    ref = oracle.scan_bwd(*(to_f64(inp[k]) for k in KEYS), to_f64(dy), **kw)
    for k in GKEYS + (("h0", "Bprev", "xprev") if with_state else ("h0",)):
        assert_err(to_f64(g[k]), ref[k], BAR, f"d{k}", floor=1e-3)


def test_backward_full_size_sampled():
    # the SISO N = 64 training shape (batch 4, 32 heads, L = 4096): two sequences against the oracle
    w = WORKLOADS["siso_n64"]
    inp = prefill_inputs(w, "cuda")
    dy = _rand(inp["x"].shape, 9)
    g = m3.scan_bwd(*(inp[k] for k in KEYS), dy)
    assert m3.device_status() == m3.M3_OK
    for b, h in ((0, 0), (w.batch - 1, w.nheads - 1)):
        one = {k: to_f64(inp[k][b:b + 1, :, h:h + 1]) for k in KEYS}
        ref = oracle.scan_bwd(*(one[k] for k in KEYS), to_f64(dy[b:b + 1, :, h:h + 1]))
        for k in GKEYS:
            assert_err(to_f64(g[k][b:b + 1, :, h:h + 1]), ref[k], BAR, f"d{k} {(b, h)}", floor=1e-3)
        assert_err(to_f64(g["h0"][b:b + 1, h:h + 1]), ref["h0"], BAR, f"dh0 {(b, h)}", floor=1e-3)


def test_backward_of_empty_sequence_passes_the_state_gradients_through():
    w = WORKLOADS["siso_n64"].with_(batch=2, nheads=3, seqlen=0)
    inp = prefill_inputs(w, "cuda")
    dh = _rand((2, 3, 64, 64), 1)
    dBo = _rand((2, 3, 1, 64), 2)
    g = m3.scan_bwd(*(inp[k] for k in KEYS), torch.empty(inp["x"].shape, device="cuda"), dh_out=dh, dB_prev_out=dBo)
    torch.cuda.synchronize()
    assert torch.equal(g["h0"], dh) and torch.equal(g["Bprev"], dBo)
    assert not torch.any(g["xprev"])
