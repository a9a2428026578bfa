"""The C-ABI library: it loads, exports every symbol include/mamba3.h declares,
and rejects bad arguments with a status code before launching anything.

These run without a GPU.  On a machine with a GPU, the pointers handed to the
library are real (tiny) device allocations, so a validation bug could never
send a kernel to a bogus address.
"""
import ctypes
import os
import re

import pytest
import torch

import selective_state_space_134_b300 as m3
from selective_state_space_134_b300 import mamba3 as api

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mamba3.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mamba3_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert {"mamba3_scan_fwd", "mamba3_decode_step", "mamba3_scan_fwd_workspace"} <= set(names)
    lib = m3.lib()
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version():
    assert m3.status_string(0) == "ok"
    for code in range(1, 6):
        assert m3.status_string(code) not in ("ok", "unknown status")
    assert m3.status_string(99) == "unknown status"
    assert m3.lib().mamba3_version() >= 100


class Ptrs:
    """16-byte aligned pointers: real device buffers when a GPU exists, else fake addresses."""

    def __init__(self):
        self.keep = []
        self.gpu = torch.cuda.is_available()
        self.fake = 0x100000

    def get(self, nbytes=4096):
        if self.gpu:
            t = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
            self.keep.append(t)
            return t.data_ptr()
        self.fake += 1 << 20
        return self.fake


def call_scan(d, ptrs, overrides=None, state_in=None, state_out=None, ws=None, ws_bytes=0):
    args = {k: ptrs.get() for k in ("x", "B", "C", "dt", "A", "lam", "theta", "y")}
    args.update(overrides or {})
    lib = m3.lib()
    return lib.mamba3_scan_fwd(ctypes.byref(d) if d is not None else None, args["x"], args["B"], args["C"], args["dt"], args["A"],
                               args["lam"], args["theta"], state_in, args["y"], state_out, ws, ws_bytes, None)


def test_workspace_query_validates():
    lib = m3.lib()
    n = ctypes.c_size_t(0)
    assert lib.mamba3_scan_fwd_workspace(None, ctypes.byref(n)) == api.M3_ERR_INVALID_ARG
    d = m3.dims(4, 4096, 32, 64, 64, 1, torch.bfloat16)
    assert lib.mamba3_scan_fwd_workspace(ctypes.byref(d), None) == api.M3_ERR_INVALID_ARG
    assert lib.mamba3_scan_fwd_workspace(ctypes.byref(d), ctypes.byref(n)) == 0
    for bad, code in [(dict(dstate=63), api.M3_ERR_UNSUPPORTED), (dict(dstate=258), api.M3_ERR_UNSUPPORTED),
                      (dict(headdim=6), api.M3_ERR_UNSUPPORTED), (dict(headdim=132), api.M3_ERR_UNSUPPORTED),
                      (dict(rank=9), api.M3_ERR_UNSUPPORTED), (dict(rank=0), api.M3_ERR_UNSUPPORTED),
                      (dict(dtype=7), api.M3_ERR_UNSUPPORTED), (dict(batch=-1), api.M3_ERR_INVALID_ARG),
                      (dict(seqlen=-5), api.M3_ERR_INVALID_ARG), (dict(nheads=0), api.M3_ERR_INVALID_ARG),
                      (dict(chunk=-1), api.M3_ERR_INVALID_ARG), (dict(ydtype=3), api.M3_ERR_UNSUPPORTED),
                      (dict(ydtype=-1), api.M3_ERR_UNSUPPORTED), (dict(dtype=api.M3_F16), api.M3_ERR_UNSUPPORTED)]:
        dd = m3.dims(4, 4096, 32, 64, 64, 1, torch.bfloat16)
        for k, v in bad.items():
            setattr(dd, k, v)
        assert lib.mamba3_scan_fwd_workspace(ctypes.byref(dd), ctypes.byref(n)) == code, bad


def test_scan_rejects_bad_pointers_before_launch():
    ptrs = Ptrs()
    before = m3.launch_count()
    d = m3.dims(1, 16, 2, 16, 16, 1, torch.float32)
    assert call_scan(None, ptrs) == api.M3_ERR_INVALID_ARG
    for k in ("x", "B", "C", "dt", "A", "lam", "theta", "y"):
        assert call_scan(d, ptrs, {k: None}) == api.M3_ERR_INVALID_ARG, k
        assert call_scan(d, ptrs, {k: ptrs.get() + 2}) == api.M3_ERR_INVALID_ARG, k   # misaligned fp32
    # state with a carry half missing
    st = api.m3_state(ptrs.get(), ptrs.get(), None)
    assert call_scan(d, ptrs, state_in=ctypes.byref(st)) == api.M3_ERR_INVALID_ARG
    assert call_scan(d, ptrs, state_out=ctypes.byref(st)) == api.M3_ERR_INVALID_ARG
    st = api.m3_state(None, None, None)
    assert call_scan(d, ptrs, state_in=ctypes.byref(st)) == api.M3_ERR_INVALID_ARG
    st = api.m3_state(ptrs.get() + 4, None, None)      # fp32 state needs 16 bytes
    assert call_scan(d, ptrs, state_in=ctypes.byref(st)) == api.M3_ERR_INVALID_ARG
    assert m3.launch_count() == before


def test_scan_requires_workspace_when_queried_nonzero():
    ptrs = Ptrs()
    d = m3.dims(1, 1 << 16, 1, 16, 16, 1, torch.float32)   # one long sequence: segmented, needs workspace
    need = m3.scan_fwd_workspace(d)
    assert need > 0
    before = m3.launch_count()
    assert call_scan(d, ptrs) == api.M3_ERR_WORKSPACE
    assert call_scan(d, ptrs, ws=ptrs.get(), ws_bytes=need - 1) == api.M3_ERR_WORKSPACE
    assert m3.launch_count() == before


def test_decode_rejects_bad_arguments_before_launch():
    ptrs = Ptrs()
    lib = m3.lib()
    before = m3.launch_count()
    d = m3.dims(2, 1, 2, 16, 16, 1, torch.bfloat16)
    good = {k: ptrs.get() for k in ("x", "B", "C", "dt", "A", "lam", "theta", "y")}

    def call(over=None, state="good"):
        a = dict(good)
        a.update(over or {})
        st = api.m3_state(ptrs.get(), ptrs.get(), ptrs.get()) if state == "good" else state
        return lib.mamba3_decode_step(ctypes.byref(d), a["x"], a["B"], a["C"], a["dt"], a["A"], a["lam"],
                                      a["theta"], ctypes.byref(st) if st is not None else None, a["y"], None)

    assert call(state=None) == api.M3_ERR_INVALID_ARG
    assert call(state=api.m3_state(ptrs.get(), None, ptrs.get())) == api.M3_ERR_INVALID_ARG
    for k in good:
        assert call({k: None}) == api.M3_ERR_INVALID_ARG, k
    dd = m3.dims(2, 1, 2, 16, 15, 1, torch.bfloat16)
    assert lib.mamba3_decode_step(ctypes.byref(dd), *[good[k] for k in ("x", "B", "C", "dt", "A", "lam", "theta")],
                                  None, good["y"], None) == api.M3_ERR_UNSUPPORTED
    assert m3.launch_count() == before


def test_pooled_decode_rejects_bad_arguments_before_launch():
    ptrs = Ptrs()
    lib = m3.lib()
    before = m3.launch_count()
    d = m3.dims(2, 1, 2, 64, 64, 4, torch.bfloat16)
    good = {k: ptrs.get() for k in ("slot", "x", "B", "C", "dt", "A", "lam", "theta", "y")}

    def call(over=None, pool="good", size=8, dd=d):
        a = dict(good)
        a.update(over or {})
        st = api.m3_state(ptrs.get(), ptrs.get(), ptrs.get()) if pool == "good" else pool
        return lib.mamba3_decode_step_pooled(ctypes.byref(dd), a["slot"], a["x"], a["B"], a["C"], a["dt"], a["A"],
                                             a["lam"], a["theta"], ctypes.byref(st) if st is not None else None,
                                             size, a["y"], None)

    assert call(pool=None) == api.M3_ERR_INVALID_ARG
    assert call(size=0) == api.M3_ERR_INVALID_ARG
    assert call(pool=api.m3_state(ptrs.get(), None, ptrs.get())) == api.M3_ERR_INVALID_ARG
    for k in good:
        assert call({k: None}) == api.M3_ERR_INVALID_ARG, k
    # shapes outside the tensor-core decode: fp32 inputs, P = 32
    assert call(dd=m3.dims(2, 1, 2, 64, 64, 4, torch.float32)) == api.M3_ERR_UNSUPPORTED
    assert call(dd=m3.dims(2, 1, 2, 32, 64, 4, torch.bfloat16)) == api.M3_ERR_UNSUPPORTED
    assert m3.launch_count() == before
    assert m3.status_string(api.M3_ERR_INDEX) == "pooled decode slot index outside the pool"


def test_grouped_bc_validation():
    lib = m3.lib()
    n = ctypes.c_size_t(0)
    # G must divide H; a negative G is an argument error
    for g in (3, -1):
        d = m3.dims(1, 64, 8, 64, 64, 1, torch.bfloat16, ngroups=g)
        assert lib.mamba3_scan_fwd_workspace(ctypes.byref(d), ctypes.byref(n)) == api.M3_ERR_INVALID_ARG
    # grouped B / C exist on the tensor-core path only: fp32 inputs or P = 32 are unsupported
    for d in (m3.dims(1, 64, 8, 64, 64, 1, torch.float32, ngroups=2),
              m3.dims(1, 64, 8, 32, 64, 1, torch.bfloat16, ngroups=2)):
        assert lib.mamba3_scan_fwd_workspace(ctypes.byref(d), ctypes.byref(n)) == api.M3_ERR_UNSUPPORTED
    d = m3.dims(1, 64, 8, 64, 64, 1, torch.bfloat16, ngroups=2)
    assert lib.mamba3_scan_fwd_workspace(ctypes.byref(d), ctypes.byref(n)) == api.M3_OK
    # decode: the same checks before any launch
    ptrs = Ptrs()
    before = m3.launch_count()
    args = [ptrs.get() for _ in range(7)]
    st = api.m3_state(ptrs.get(), ptrs.get(), ptrs.get())
    for d, want in ((m3.dims(2, 1, 8, 64, 64, 1, torch.bfloat16, ngroups=3), api.M3_ERR_INVALID_ARG),
                    (m3.dims(2, 1, 8, 64, 64, 1, torch.float32, ngroups=2), api.M3_ERR_UNSUPPORTED),
                    (m3.dims(2, 1, 8, 16, 64, 1, torch.bfloat16, ngroups=2), api.M3_ERR_UNSUPPORTED)):
        assert lib.mamba3_decode_step(ctypes.byref(d), *args, ctypes.byref(st), ptrs.get(), None) == want
    assert m3.launch_count() == before


def test_staged_prefill_rejects_bad_arguments_before_any_copy():
    lib = m3.lib()
    d = m3.dims(2, 16, 2, 64, 64, 1, torch.bfloat16)
    n = ctypes.c_size_t(0)
    assert lib.mamba3_scan_fwd_staged_workspace(ctypes.byref(d), 0, ctypes.byref(n)) == api.M3_ERR_INVALID_ARG
    assert lib.mamba3_scan_fwd_staged_workspace(ctypes.byref(d), 4, ctypes.byref(n)) == api.M3_OK
    ins = api.m3_token_inputs(*([None] * 7))
    before = m3.launch_count()
    # no input tables / zero slices / h copy without a device state
    assert lib.mamba3_scan_fwd_staged(ctypes.byref(d), None, None, None, None, None, None, None, None, 0, 1,
                                      None, None) == api.M3_ERR_INVALID_ARG
    assert lib.mamba3_scan_fwd_staged(ctypes.byref(d), ctypes.byref(ins), ctypes.byref(ins), None, None, None,
                                      None, None, None, 0, 0, None, None) == api.M3_ERR_INVALID_ARG
    assert lib.mamba3_scan_fwd_staged(ctypes.byref(d), ctypes.byref(ins), ctypes.byref(ins), None, None, None,
                                      None, 0x1000, None, 0, 1, None, None) == api.M3_ERR_INVALID_ARG
    # several token ranges need a device state (with its carry) to hand on
    assert lib.mamba3_scan_fwd_staged(ctypes.byref(d), ctypes.byref(ins), ctypes.byref(ins), None, None, None,
                                      None, None, None, 0, 2, None, None) == api.M3_ERR_INVALID_ARG
    assert m3.launch_count() == before


def test_bc_norm_validation():
    # eps < 0 or NaN, or a misaligned gain pointer: M3_ERR_INVALID_ARG before any launch; grouped
    # decode with BC normalisation: M3_ERR_UNSUPPORTED
    lib = m3.lib()
    ptrs = Ptrs()
    d = m3.dims(1, 64, 8, 64, 64, 1, torch.bfloat16)
    args = [ptrs.get() for _ in range(8)]
    before = m3.launch_count()
    for eps, wptr in ((-1.0, None), (float("nan"), None), (1e-5, ptrs.get() + 2)):
        bc = api.m3_bc_norm(wptr, None, None, None, eps)
        rc = lib.mamba3_scan_fwd_bc(ctypes.byref(d), *args[:7], ctypes.byref(bc), None, args[7], None, None, 0, None)
        assert rc == api.M3_ERR_INVALID_ARG, eps
        st = api.m3_state(ptrs.get(), ptrs.get(), ptrs.get())
        rc = lib.mamba3_decode_step_bc(ctypes.byref(d), *args[:7], ctypes.byref(bc), ctypes.byref(st), args[7], None)
        assert rc == api.M3_ERR_INVALID_ARG, eps
    bc = api.m3_bc_norm(None, None, None, None, 1e-5)
    dg = m3.dims(1, 1, 8, 64, 64, 1, torch.bfloat16, ngroups=2)
    st = api.m3_state(ptrs.get(), ptrs.get(), ptrs.get())
    rc = lib.mamba3_decode_step_bc(ctypes.byref(dg), *args[:7], ctypes.byref(bc), ctypes.byref(st), args[7], None)
    assert rc == api.M3_ERR_UNSUPPORTED
    assert m3.launch_count() == before


def test_backward_validation():
    lib = m3.lib()
    ptrs = Ptrs()
    n = ctypes.c_size_t(0)
    d = m3.dims(2, 100, 4, 64, 64, 1, torch.bfloat16)
    assert lib.mamba3_scan_bwd_workspace(ctypes.byref(d), ctypes.byref(n)) == 0 and n.value > 0
    # one B and C per head only; N * P <= 8192
    for bad in (m3.dims(2, 100, 4, 64, 64, 1, torch.bfloat16, ngroups=2), m3.dims(2, 100, 4, 128, 128, 1, torch.float32)):
        assert lib.mamba3_scan_bwd_workspace(ctypes.byref(bad), ctypes.byref(n)) == api.M3_ERR_UNSUPPORTED
    ins = api.m3_token_inputs(*(ptrs.get() for _ in range(7)))
    gin = api.m3_grads_in(ptrs.get(), None, None, None)
    gout = api.m3_grads_out(*(ptrs.get() for _ in range(7)), None, None, None)
    before = m3.launch_count()
    # missing workspace, missing dy, missing dx, NULL structs
    assert lib.mamba3_scan_bwd(ctypes.byref(d), ctypes.byref(ins), None, ctypes.byref(gin), ctypes.byref(gout),
                               None, 0, None) == api.M3_ERR_WORKSPACE
    ws = ptrs.get(n.value)
    gin0 = api.m3_grads_in(None, None, None, None)
    assert lib.mamba3_scan_bwd(ctypes.byref(d), ctypes.byref(ins), None, ctypes.byref(gin0), ctypes.byref(gout),
                               ws, n.value, None) == api.M3_ERR_INVALID_ARG
    gout0 = api.m3_grads_out(None, *(ptrs.get() for _ in range(6)), None, None, None)
    assert lib.mamba3_scan_bwd(ctypes.byref(d), ctypes.byref(ins), None, ctypes.byref(gin), ctypes.byref(gout0),
                               ws, n.value, None) == api.M3_ERR_INVALID_ARG
    assert lib.mamba3_scan_bwd(ctypes.byref(d), None, None, ctypes.byref(gin), ctypes.byref(gout),
                               ws, n.value, None) == api.M3_ERR_INVALID_ARG
    assert m3.launch_count() == before


def test_long_prefill_plan_cuts_the_state_pass_into_full_waves():
    # The tensor-core plan of the long-context workload (64 sequences of 131072 tokens, N = 128, R = 4)
    # on 148 SMs: two segments, the first cut into the smallest number of whole pieces that minimises
    # waves / pieces (16 pieces: 1024 CTAs in 7 waves, 0.4375 of a segment per CTA slot, against 0.5
    # for one wave of 2 pieces), so the workspace holds (2 - 1) * 16 + 1 = 17 state slots per sequence
    # and the segment totals of 16 pieces.  (The workspace query covers the SIMT plan too; here it has
    # 5 segments and needs less.)
    if torch.cuda.is_available() and torch.cuda.get_device_properties(0).multi_processor_count != 148:
        pytest.skip("the plan is pinned for 148 SMs")
    lib = m3.lib()
    n = ctypes.c_size_t(0)
    d = m3.dims(1, 131072, 64, 64, 128, 4, torch.bfloat16)
    assert lib.mamba3_scan_fwd_workspace(ctypes.byref(d), ctypes.byref(n)) == 0
    bh, N, P, slots = 64, 128, 64, 17
    state = bh * slots * N * P * 4
    tot = bh * (slots - 1) * (1 + N // 2) * 4
    assert n.value == ((state + 255) // 256) * 256 + tot
