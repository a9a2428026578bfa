"""mamba3_scan_fwd_noalloc, the prefill for callers that cannot allocate device
memory (an engine that owns every allocation, a latency-critical path that
cannot take cudaMalloc's synchronisation, a plain C caller without an
allocator): it must give the same results as mamba3_scan_fwd with a
caller-provided workspace, call after call, although every call reuses the
library's one static scratch array, and it must refuse problems whose scratch
need exceeds that array before launching anything.

This file is collected last on purpose; it passes alone in a fresh process and
after the other tests.
"""
import ctypes

import pytest
import torch

import selective_state_space_134_b300 as m3
from selective_state_space_134_b300 import mamba3 as api
from selective_state_space_134_b300.synth import WORKLOADS, prefill_inputs
from helpers import KEYS

pytestmark = pytest.mark.gpu

LIMIT = 16 << 20   # M3_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_134_b300 import build
    build.build()


def _run(fn, inp, w, **kw):
    st = m3.State.zeros(w.batch, w.nheads, w.P, w.N, w.R, inp["x"].dtype)
    y = fn(*(inp[k] for k in KEYS), state_out=st, **kw)
    assert m3.device_status() == m3.M3_OK
    return y, st


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    # few long sequences: the prefill is split into segments and needs scratch
    w1 = WORKLOADS["long_n128_r4"].with_(batch=1, nheads=2, seqlen=3000)
    w2 = WORKLOADS["mimo_r4"].with_(batch=1, nheads=3, seqlen=2500, seed=9)
    for w in (w1, w2):
        need = m3.scan_fwd_workspace(m3.dims(w.batch, w.seqlen, w.nheads, w.P, w.N, w.R, torch.bfloat16))
        assert 0 < need <= LIMIT
    calls = [(w1, prefill_inputs(w1, "cuda")), (w2, prefill_inputs(w2, "cuda"))]
    # Two different problems back to back: leftovers in the shared scratch must not matter.  Both
    # entry points run the same plan and the same deterministic kernels (no atomics, fixed
    # reduction orders); only the scratch address differs, so the results must be bit-identical.
    for w, inp in calls:
        y_ref, s_ref = _run(m3.scan_fwd, inp, w)
        y, s = _run(api.scan_fwd_noalloc, inp, w)
        assert torch.equal(y, y_ref)
        assert torch.equal(s.h, s_ref.h)
        assert torch.equal(s.B_prev, s_ref.B_prev) and torch.equal(s.x_prev, s_ref.x_prev)


def test_noalloc_rejects_problems_beyond_the_static_scratch():
    # 2 sequences of 37888 tokens with N = P = 128: the segment states need ~19 MB > 16 MiB
    w = WORKLOADS["siso_n128"].with_(batch=1, nheads=2, seqlen=37888, P=128)
    d = m3.dims(w.batch, w.seqlen, w.nheads, w.P, w.N, w.R, torch.bfloat16)
    assert m3.scan_fwd_workspace(d) > LIMIT
    inp = prefill_inputs(w, "cuda")
    y = torch.empty(inp["x"].shape, dtype=torch.float32, device="cuda")
    before = m3.launch_count()
    fn = m3.lib().mamba3_scan_fwd_noalloc
    fn.argtypes = [ctypes.POINTER(api.m3_dims)] + [ctypes.c_void_p] * 7 + \
        [ctypes.POINTER(api.m3_state), ctypes.c_void_p, ctypes.POINTER(api.m3_state), ctypes.c_void_p]
    fn.restype = ctypes.c_int
    rc = fn(ctypes.byref(d), *(inp[k].data_ptr() for k in KEYS), None, y.data_ptr(), None, None)
    assert rc == api.M3_ERR_WORKSPACE
    assert m3.launch_count() == before
