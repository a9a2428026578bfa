"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Metric: max|y - y_ref| / rms(y_ref) (and the same for the final state), with
the tolerances of the Mamba-3 recurrence study: 1e-4 for fp32 inputs, 2e-2 for
bf16 inputs (fp32 state on the GPU in both cases).  Small cases compare every
element; full-size workloads compare sampled (b, h) sequences, which the
oracle computes one by one on the same inputs.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_134_b300 as m3
from selective_state_space_134_b300.synth import WORKLOADS, decode_pool, decode_state, prefill_inputs, to_f64
from helpers import KEYS, TOL, assert_err, norm_err, oracle_full, oracle_slices

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_134_b300 import build
    build.build()
    torch.cuda.init()


def gpu_scan(inp, state_in=None, chunk=0, carry_out=True, inplace=False):
    x = inp["x"]
    b, L, H, R, P = x.shape
    N = inp["B"].shape[-1]
    if inplace:
        st_out = state_in
    else:
        st_out = m3.State.zeros(b, H, P, N, R, x.dtype) if carry_out else \
            m3.State(torch.zeros(b, H, N, P, device="cuda"))
    y = m3.scan_fwd(*(inp[k] for k in KEYS), state_in=state_in, state_out=st_out, chunk=chunk)
    assert m3.device_status() == m3.M3_OK
    torch.cuda.synchronize()
    return y, st_out


def random_state(b, H, P, N, R, dtype, seed=0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return m3.State(torch.randn(b, H, N, P, device="cuda", generator=g),
                    torch.randn(b, H, R, N, device="cuda", generator=g).to(dtype),
                    torch.randn(b, H, R, P, device="cuda", generator=g).to(dtype))


SMALL = {
    # name: (workload, overrides)
    "tiny_f32": ("tiny_f32", {}),
    "siso_n64_small": ("siso_n64", dict(batch=2, nheads=3, seqlen=300)),
    "siso_n128_small": ("siso_n128", dict(batch=1, nheads=2, seqlen=333)),
    "mimo_r4_small": ("mimo_r4", dict(batch=1, nheads=3, seqlen=201)),
    "long_small_segmented": ("long_n128_r4", dict(batch=1, nheads=2, seqlen=1100)),
    "siso_n64_small_f32": ("siso_n64", dict(batch=1, nheads=2, seqlen=300, dtype="f32")),
    "mimo_r4_small_f32_segmented": ("mimo_r4", dict(batch=1, nheads=1, seqlen=777, dtype="f32")),
    "odd_shapes_f32": ("tiny_f32", dict(N=2, P=4, R=3, seqlen=37, nheads=3)),
    "odd_shapes_bf16": ("tiny_f32", dict(N=6, P=8, R=2, seqlen=65, nheads=2, dtype="bf16")),
    "single_token": ("siso_n64", dict(batch=2, nheads=2, seqlen=1)),
}


@pytest.mark.parametrize("case", sorted(SMALL))
@pytest.mark.parametrize("with_state", [False, True])
def test_scan_small_matches_oracle(case, with_state):
    wname, over = SMALL[case]
    w = WORKLOADS[wname].with_(**over)
    inp = prefill_inputs(w, "cuda")
    st = random_state(w.batch, w.nheads, w.P, w.N, w.R, inp["x"].dtype) if with_state else None
    y, so = gpu_scan(inp, state_in=st)
    yr, hr, Br, xr = oracle_full(inp, st)
    tol = TOL[w.dtype]
    assert_err(to_f64(y), yr, tol, "y")
    assert_err(to_f64(so.h), hr, tol, "h")
    np.testing.assert_array_equal(to_f64(so.B_prev), Br)     # carry is a plain copy
    np.testing.assert_array_equal(to_f64(so.x_prev), xr)


@pytest.mark.parametrize("wname", ["siso_n64", "siso_n128", "mimo_r4", "long_n128_r4"])
def test_scan_full_size_sampled(wname):
    w = WORKLOADS[wname]
    inp = prefill_inputs(w, "cuda")
    y, so = gpu_scan(inp)
    pairs = [(0, 0), (w.batch - 1, w.nheads - 1)] if wname == "long_n128_r4" else \
        [(0, 0), (w.batch // 2, w.nheads // 3), (w.batch - 1, w.nheads - 1)]
    # oracle: all sampled sequences stacked along the batch axis, one thread each
    stack = {k: torch.cat([inp[k][b:b + 1, :, h:h + 1] for b, h in pairs], dim=0) for k in KEYS}
    yr, hr, _, _ = oracle.scan(*(to_f64(stack[k]) for k in KEYS), nthreads=len(pairs))
    for i, (b, h) in enumerate(pairs):
        assert_err(to_f64(y[b:b + 1, :, h:h + 1]), yr[i:i + 1], TOL[w.dtype], f"y (b, h) = {(b, h)}")
        assert_err(to_f64(so.h[b:b + 1, h:h + 1]), hr[i:i + 1], TOL[w.dtype], f"h (b, h) = {(b, h)}")
    assert torch.isfinite(y.float()).all()


def _random_shapes(n, seed=2026):
    import random
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        N, R = rng.choice([64, 128]), rng.choice([1, 2, 4, 8])
        H, b = rng.randint(1, 40), rng.randint(1, 2)
        L = rng.randint(1, 1400)
        out.append((N, R, H, b, L, rng.random() < 0.5))
    return out


@pytest.mark.parametrize("N,R,H,b,L,with_state", _random_shapes(8))
def test_prefill_random_shapes_match_oracle(N, R, H, b, L, with_state):
    # seeded shapes over the planner's cases: one or several segments, state-pass pieces,
    # ragged last chunks and segments, every rank; all sequences against the oracle
    w = WORKLOADS["mimo_r4"].with_(batch=b, nheads=H, seqlen=L, N=N, R=R)
    inp = prefill_inputs(w, "cuda")
    st = random_state(b, H, w.P, N, R, inp["x"].dtype, seed=L) if with_state else None
    y, so = gpu_scan(inp, state_in=st)
    yr, hr, Br, xr = oracle_full(inp, st)
    assert_err(to_f64(y), yr, TOL[w.dtype], "y")
    assert_err(to_f64(so.h), hr, TOL[w.dtype], "h")
    np.testing.assert_array_equal(to_f64(so.B_prev), Br)
    np.testing.assert_array_equal(to_f64(so.x_prev), xr)


@pytest.mark.parametrize("with_state", [False, True])
def test_segmented_prefill_with_state_pass_pieces(with_state):
    # 64 sequences, L = 1000, N = 128, R = 4 (16-token chunks): two segments of 512 tokens
    # (one wave of CTAs), the state pass cut into two pieces of 256 tokens, a ragged last
    # segment; every sequence against the oracle
    w = WORKLOADS["long_n128_r4"].with_(batch=1, nheads=64, seqlen=1000)
    inp = prefill_inputs(w, "cuda")
    st = random_state(w.batch, w.nheads, w.P, w.N, w.R, inp["x"].dtype) if with_state else None
    y, so = gpu_scan(inp, state_in=st)
    yr, hr, Br, xr = oracle_full(inp, st)
    assert_err(to_f64(y), yr, TOL[w.dtype], "y")
    assert_err(to_f64(so.h), hr, TOL[w.dtype], "h")
    np.testing.assert_array_equal(to_f64(so.B_prev), Br)
    np.testing.assert_array_equal(to_f64(so.x_prev), xr)


@pytest.mark.parametrize("wname", ["decode_n64_r1", "decode_n64_r4", "decode_n128_r1", "decode_n128_r4"])
def test_decode_full_size_matches_oracle(wname):
    w = WORKLOADS[wname]
    st = decode_state(w, "cuda")
    state = m3.State(st["h"].clone(), st["B_prev"].clone(), st["x_prev"].clone())
    pool = decode_pool(w, "cuda", pool=3)
    ref_h, ref_B, ref_x = to_f64(st["h"]), to_f64(st["B_prev"]), to_f64(st["x_prev"])
    for step, tok in enumerate(pool):
        y = m3.decode_step(*(tok[k] for k in KEYS), state=state)
        assert m3.device_status() == m3.M3_OK
        yr, ref_h, ref_B, ref_x = oracle.decode_step(*(to_f64(tok[k]) for k in KEYS), ref_h, ref_B, ref_x)
        assert_err(to_f64(y), yr, TOL[w.dtype], f"y {step}")
        assert_err(to_f64(state.h), ref_h, 1e-5, f"h step {step}")      # fp32 state, exact-input update
        np.testing.assert_array_equal(to_f64(state.B_prev), ref_B)
        np.testing.assert_array_equal(to_f64(state.x_prev), ref_x)


@pytest.mark.parametrize("R,N,H", [(1, 64, 45), (2, 64, 45), (8, 64, 45), (4, 64, 45), (1, 64, 46), (2, 64, 46),
                                   (8, 64, 46), (1, 128, 45), (2, 128, 45), (8, 128, 45)])
def test_decode_tensor_core_ranks_match_oracle(R, N, H):
    # bf16, P = 64: the tensor-core decode; 7 x 45 = 315 heads (one head per unit) and
    # 7 x 46 = 322 heads (N = 64: two heads per unit) leave a ragged last round of units
    w = WORKLOADS["decode_n64_r4"].with_(batch=7, nheads=H, N=N, R=R)
    st = decode_state(w, "cuda")
    state = m3.State(st["h"].clone(), st["B_prev"].clone(), st["x_prev"].clone())
    ref_h, ref_B, ref_x = to_f64(st["h"]), to_f64(st["B_prev"]), to_f64(st["x_prev"])
    for step, tok in enumerate(decode_pool(w, "cuda", pool=2)):
        y = m3.decode_step(*(tok[k] for k in KEYS), state=state)
        assert m3.device_status() == m3.M3_OK
        yr, ref_h, ref_B, ref_x = oracle.decode_step(*(to_f64(tok[k]) for k in KEYS), ref_h, ref_B, ref_x)
        assert_err(to_f64(y), yr, 1e-4, f"y step {step}")     # hi + lo split of h: far inside the bf16 bar
        assert_err(to_f64(state.h), ref_h, 1e-5, f"h {step}")
        np.testing.assert_array_equal(to_f64(state.B_prev), ref_B)
        np.testing.assert_array_equal(to_f64(state.x_prev), ref_x)


@pytest.mark.parametrize("N,R,H", [(64, 4, 8), (64, 1, 8), (128, 4, 8), (64, 8, 5)])
def test_decode_pooled_matches_oracle(N, R, H):
    # six batch rows on a pool of 11 states: active rows name distinct slots, two rows are
    # inactive (-1); H = 8 pairs adjacent heads for N = 64, H = 5 keeps one head per unit
    S = 11
    slots = [7, -1, 0, 10, 3, -1]
    w = WORKLOADS["decode_n64_r4"].with_(batch=len(slots), nheads=H, N=N, R=R)
    ps = decode_state(w.with_(batch=S), "cuda")
    pool = m3.State(ps["h"].clone(), ps["B_prev"].clone(), ps["x_prev"].clone())
    tok = decode_pool(w, "cuda", pool=1)[0]
    slot = torch.tensor(slots, dtype=torch.int32, device="cuda")
    y = torch.full((w.batch, H, R, w.P), 12345.0, device="cuda")
    m3.decode_step_pooled(*(tok[k] for k in KEYS), slot=slot, pool=pool, y=y)
    assert m3.device_status() == m3.M3_OK
    for b, sl in enumerate(slots):
        if sl < 0:
            assert bool((y[b] == 12345.0).all()), b          # inactive row: y untouched
            continue
        one = {k: to_f64(tok[k][b:b + 1]) for k in KEYS}
        yr, hr, Br, xr = oracle.decode_step(*(one[k] for k in KEYS), to_f64(ps["h"][sl:sl + 1]),
                                            to_f64(ps["B_prev"][sl:sl + 1]), to_f64(ps["x_prev"][sl:sl + 1]))
        assert_err(to_f64(y[b:b + 1]), yr, 1e-4, f"y {b}")
        assert_err(to_f64(pool.h[sl:sl + 1]), hr, 1e-5, f"h {b}")
        np.testing.assert_array_equal(to_f64(pool.B_prev[sl:sl + 1]), Br)
        np.testing.assert_array_equal(to_f64(pool.x_prev[sl:sl + 1]), xr)
    for sl in set(range(S)) - set(slots):                          # slots no row names: bitwise unchanged
        assert torch.equal(pool.h[sl], ps["h"][sl]) and torch.equal(pool.B_prev[sl], ps["B_prev"][sl])
        assert torch.equal(pool.x_prev[sl], ps["x_prev"][sl])


def test_decode_pooled_slot_outside_pool_is_reported_and_skipped():
    # the kernel checks every slot against the pool size before touching the pool
    S = 4
    w = WORKLOADS["decode_n64_r4"].with_(batch=3, nheads=4, N=64, R=4)
    ps = decode_state(w.with_(batch=S), "cuda")
    pool = m3.State(ps["h"].clone(), ps["B_prev"].clone(), ps["x_prev"].clone())
    tok = decode_pool(w, "cuda", pool=1)[0]
    slot = torch.tensor([2, S, 0], dtype=torch.int32, device="cuda")
    y = torch.full((3, 4, 4, 64), -7.0, device="cuda")
    m3.decode_step_pooled(*(tok[k] for k in KEYS), slot=slot, pool=pool, y=y)
    assert m3.device_status() == m3.M3_ERR_INDEX
    assert m3.device_status() == m3.M3_OK                          # read and cleared
    assert bool((y[1] == -7.0).all())
    assert torch.equal(pool.h[1], ps["h"][1]) and torch.equal(pool.h[3], ps["h"][3])
    assert not torch.equal(pool.h[2], ps["h"][2])                  # the valid rows ran


def _grouped(t, H, G, axis):
    # B / C shared by groups of H / G heads: the first head's values of every group, and the
    # per-head expansion the oracle reads (head h takes group h // (H / G))
    idx = torch.arange(0, H, H // G, device=t.device)
    g = t.index_select(axis, idx).contiguous()
    return g, g.repeat_interleave(H // G, dim=axis)


@pytest.mark.parametrize("wname,H,G,L", [("siso_n64", 8, 2, 700), ("siso_n64", 4, 1, 300),
                                         ("long_n128_r4", 6, 3, 900), ("mimo_r4", 40, 8, 260)])
def test_prefill_grouped_bc_matches_oracle(wname, H, G, L):
    # grouped B / C (G groups of H / G heads) on the tensor-core prefill, one or several
    # segments, with an initial state; against the oracle on the per-head expansion
    w = WORKLOADS[wname].with_(batch=2, nheads=H, seqlen=L)
    inp = prefill_inputs(w, "cuda")
    full = dict(inp)
    for k in ("B", "C"):
        inp[k], full[k] = _grouped(inp[k], H, G, 2)
    st = random_state(w.batch, H, w.P, w.N, w.R, inp["x"].dtype, seed=G)
    y, so = gpu_scan(inp, state_in=st)
    yr, hr, Br, xr = oracle_full(full, st)
    assert_err(to_f64(y), yr, TOL[w.dtype], "y")
    assert_err(to_f64(so.h), hr, TOL[w.dtype], "h")
    np.testing.assert_array_equal(to_f64(so.B_prev), Br)       # per-head carry of the group's B
    np.testing.assert_array_equal(to_f64(so.x_prev), xr)


@pytest.mark.parametrize("N,R,H,G", [(64, 4, 8, 2), (64, 1, 8, 4), (128, 4, 6, 1), (64, 8, 8, 8)])
def test_decode_grouped_bc_matches_oracle(N, R, H, G):
    w = WORKLOADS["decode_n64_r4"].with_(batch=5, nheads=H, N=N, R=R)
    st = decode_state(w, "cuda")
    state = m3.State(st["h"].clone(), st["B_prev"].clone(), st["x_prev"].clone())
    ref_h, ref_B, ref_x = to_f64(st["h"]), to_f64(st["B_prev"]), to_f64(st["x_prev"])
    for step, tok in enumerate(decode_pool(w, "cuda", pool=2)):
        full = dict(tok)
        for k in ("B", "C"):
            tok[k], full[k] = _grouped(tok[k], H, G, 1)
        y = m3.decode_step(*(tok[k] for k in KEYS), state=state)
        assert m3.device_status() == m3.M3_OK
        yr, ref_h, ref_B, ref_x = oracle.decode_step(*(to_f64(full[k]) for k in KEYS), ref_h, ref_B, ref_x)
        assert_err(to_f64(y), yr, 1e-4, f"y {step}")
        assert_err(to_f64(state.h), ref_h, 1e-5, f"h {step}")
        np.testing.assert_array_equal(to_f64(state.B_prev), ref_B)
        np.testing.assert_array_equal(to_f64(state.x_prev), ref_x)


@pytest.mark.parametrize("dtype,P,N,R,b,H", [
    ("f32", 64, 64, 1, 5, 67), ("f32", 64, 64, 4, 5, 67), ("f32", 64, 128, 4, 3, 41), ("f32", 64, 64, 2, 2, 9),
    ("f32", 64, 128, 8, 2, 7), ("f32", 32, 64, 4, 4, 37), ("f32", 128, 32, 2, 3, 19), ("f32", 64, 48, 1, 2, 11),
    ("bf16", 128, 64, 1, 5, 33), ("bf16", 128, 128, 4, 2, 21), ("bf16", 32, 64, 2, 4, 37), ("bf16", 32, 32, 8, 3, 9),
    ("bf16", 64, 96, 4, 2, 19)])
def test_decode_streaming_kernel_matches_oracle(dtype, P, N, R, b, H):
    # fp32 inputs with P in {32, 64, 128}, and bf16 inputs outside the tensor-core shapes, go to the
    # streaming FMA kernel; its arithmetic is fp32 on exactly the stored inputs, so y and h match the
    # fp64 oracle to fp32 rounding over several steps
    w = WORKLOADS["decode_n64_r4"].with_(batch=b, nheads=H, P=P, N=N, R=R, dtype=dtype)
    st = decode_state(w, "cuda")
    state = m3.State(st["h"].clone(), st["B_prev"].clone(), st["x_prev"].clone())
    ref_h, ref_B, ref_x = to_f64(st["h"]), to_f64(st["B_prev"]), to_f64(st["x_prev"])
    for step, tok in enumerate(decode_pool(w, "cuda", pool=3)):
        y = m3.decode_step(*(tok[k] for k in KEYS), state=state)
        assert m3.decode_last_variant() == m3.DECODE_STREAM
        assert m3.device_status() == m3.M3_OK
        yr, ref_h, ref_B, ref_x = oracle.decode_step(*(to_f64(tok[k]) for k in KEYS), ref_h, ref_B, ref_x)
        assert_err(to_f64(y), yr, 1e-5, f"y {step}")
        assert_err(to_f64(state.h), ref_h, 1e-5, f"h {step}")
        np.testing.assert_array_equal(to_f64(state.B_prev), ref_B)
        np.testing.assert_array_equal(to_f64(state.x_prev), ref_x)


def test_decode_variants_are_selected_by_shape():
    # the bench's bf16 P = 64 workloads take the tensor-core kernel; P = 16 the generic one
    for over, want in ((dict(), m3.DECODE_TENSOR), (dict(P=16, dtype="f32"), m3.DECODE_GENERIC),
                       (dict(dtype="f32"), m3.DECODE_STREAM)):
        w = WORKLOADS["decode_n64_r4"].with_(batch=2, nheads=4, **over)
        st = decode_state(w, "cuda")
        state = m3.State(st["h"], st["B_prev"], st["x_prev"])
        tok = decode_pool(w, "cuda", pool=1)[0]
        m3.decode_step(*(tok[k] for k in KEYS), state=state)
        assert m3.decode_last_variant() == want, over


def test_decode_f32_tight():
    w = WORKLOADS["tiny_f32"].with_(batch=3, nheads=5, N=32, P=16, R=2)
    st = decode_state(w, "cuda")
    state = m3.State(st["h"].clone(), st["B_prev"].clone(), st["x_prev"].clone())
    tok = decode_pool(w, "cuda", pool=1)[0]
    y = m3.decode_step(*(tok[k] for k in KEYS), state=state)
    yr, hr, _, _ = oracle.decode_step(*(to_f64(tok[k]) for k in KEYS), to_f64(st["h"]), to_f64(st["B_prev"]),
                                      to_f64(st["x_prev"]))
    assert_err(to_f64(y), yr, 1e-5, "y")
    assert_err(to_f64(state.h), hr, 1e-5, "h")


# ---------------------------------------------------------------- GPU-side invariants

def test_chunk_length_does_not_change_the_result():
    w = WORKLOADS["mimo_r4"].with_(batch=1, nheads=2, seqlen=150, dtype="f32", R=2)
    inp = prefill_inputs(w, "cuda")
    ys = [gpu_scan(inp, chunk=q)[0] for q in (0, 1, 7, 32, 64)]
    for y in ys[1:]:
        assert_err(to_f64(y), to_f64(ys[0]), 1e-5, "y")


def test_split_prefill_and_decode_resume_equal_full_prefill():
    w = WORKLOADS["siso_n64"].with_(batch=2, nheads=2, seqlen=200)
    inp = prefill_inputs(w, "cuda")
    y_full, s_full = gpu_scan(inp)
    L1 = 77
    first = {k: v[:, :L1].contiguous() for k, v in inp.items()}
    rest = {k: v[:, L1:].contiguous() for k, v in inp.items()}
    y1, s1 = gpu_scan(first)
    y2, s2 = gpu_scan(rest, state_in=s1)
    tol = TOL[w.dtype]
    assert_err(to_f64(torch.cat([y1, y2], 1)), to_f64(y_full), tol, "y")
    assert_err(to_f64(s2.h), to_f64(s_full.h), tol, "h")
    # prefill L - k tokens, then k decode steps
    k = 5
    head = {kk: v[:, :-k].contiguous() for kk, v in inp.items()}
    _, st = gpu_scan(head)
    for t in range(w.seqlen - k, w.seqlen):
        yt = m3.decode_step(*(inp[kk][:, t].contiguous() for kk in KEYS), state=st)
        assert_err(to_f64(yt), to_f64(y_full[:, t]), tol, "y")
    assert_err(to_f64(st.h), to_f64(s_full.h), tol, "h")


@pytest.mark.parametrize("wname,over", [("siso_n64", dict(batch=3, nheads=4)), ("mimo_r4", dict(batch=2, nheads=3)),
                                        ("siso_n128", dict(batch=2, nheads=3))])
def test_alternating_prefill_and_decode_on_one_stream_match_oracle(wname, over):
    # prefill pieces and single decode steps alternate on one stream with no host synchronisation
    # between the calls: each call reads the state the call before wrote (the kernels are launched
    # as programmatic dependents and must wait for it), in both orders (prefill after decode and
    # decode after prefill); every output and the final state against the oracle
    pieces = [70, 3, 45, 1, 1, 60, 2]   # tokens per call: prefill for >= 3 (ragged chunks), else decode steps
    w = WORKLOADS[wname].with_(seqlen=sum(pieces), **over)
    inp = prefill_inputs(w, "cuda")
    st = m3.State.zeros(w.batch, w.nheads, w.P, w.N, w.R, inp["x"].dtype)
    ys, t = [], 0
    for n in pieces:
        if n >= 3:
            part = {k: v[:, t:t + n].contiguous() for k, v in inp.items()}
            ys.append(m3.scan_fwd(*(part[k] for k in KEYS), state_in=st, state_out=st))
        else:
            for i in range(n):
                ys.append(m3.decode_step(*(inp[k][:, t + i].contiguous() for k in KEYS), state=st).unsqueeze(1))
        t += n
    assert m3.device_status() == m3.M3_OK
    torch.cuda.synchronize()
    yr, hr, bpr, xpr = oracle_full(inp)
    tol = TOL[w.dtype]
    assert_err(to_f64(torch.cat(ys, dim=1)), yr, tol, "y")
    assert_err(to_f64(st.h), hr, tol, "h")
    assert np.array_equal(to_f64(st.B_prev), bpr) and np.array_equal(to_f64(st.x_prev), xpr)


@pytest.mark.parametrize("wname,over", [("siso_n64", dict(nheads=2, seqlen=129)), ("siso_n128", dict(nheads=2, seqlen=65)),
                                        ("mimo_r4", dict(nheads=2, seqlen=33)),
                                        ("long_n128_r4", dict(nheads=2, seqlen=1041))])
def test_last_chunk_sees_nothing_of_the_next_sequence(wname, over):
    # Sequences whose last chunk holds one token (or a few); the batch row after the first one
    # starts with B, C and x set to +inf.  The tensor-core prefill's input tiles end at each
    # sequence's last token, so none of those values may reach the first row's last chunk: a value
    # read past the end would turn into NaN (a zero weight times inf) in its scores, its state or its
    # tile scales, where the oracle, which sees each sequence alone, has finite results.  The planted
    # row's own outputs are not compared (they are not finite); the rows before and after it are
    w = WORKLOADS[wname].with_(batch=3, **over)
    inp = prefill_inputs(w, "cuda")
    for k in ("B", "C", "x"):
        v = inp[k].float()
        v[1, :8] = float("inf")
        inp[k] = v.to(inp[k].dtype)
    y, so = gpu_scan(inp)
    yr, hr, Br, xr = oracle_full(inp)
    tol = TOL[w.dtype]
    for b in (0, 2):
        assert_err(to_f64(y[b:b + 1]), yr[b:b + 1], tol, f"y batch {b}")
        assert_err(to_f64(so.h[b:b + 1]), hr[b:b + 1], tol, f"h batch {b}")
    np.testing.assert_array_equal(to_f64(so.B_prev), Br)
    np.testing.assert_array_equal(to_f64(so.x_prev), xr)


def test_in_place_state_update_equals_out_of_place():
    w = WORKLOADS["siso_n64"].with_(batch=2, nheads=3, seqlen=130)
    inp = prefill_inputs(w, "cuda")
    st = random_state(w.batch, w.nheads, w.P, w.N, w.R, inp["x"].dtype, seed=3)
    st_copy = m3.State(st.h.clone(), st.B_prev.clone(), st.x_prev.clone())
    y1, s1 = gpu_scan(inp, state_in=st_copy)
    y2, s2 = gpu_scan(inp, state_in=st, inplace=True)
    assert torch.equal(y1, y2)
    assert torch.equal(s1.h, st.h) and torch.equal(s1.B_prev, st.B_prev) and torch.equal(s1.x_prev, st.x_prev)


@pytest.mark.parametrize("R,L", [(1, 1728), (2, 864), (4, 432), (8, 216)])
def test_state_pass_pieces_ending_inside_a_chunk(R, L):
    # N = 128: the state pass runs chunks of 128 rows, twice the output pass's 64.  An even split of
    # these lengths over the segments would give pieces of 7 output chunks, half a state-pass chunk
    # past a whole number of them; a CTA starts at a whole chunk, so the plan must cut the segments at
    # whole state-pass chunks (a piece starting inside one re-adds that chunk's first tokens and
    # corrupts every later segment's start state).  h0 and the carry in, every output against the oracle
    w = WORKLOADS["long_n128_r4"].with_(batch=1, nheads=3, seqlen=L, R=R)
    inp = prefill_inputs(w, "cuda")
    st = random_state(w.batch, w.nheads, w.P, w.N, w.R, inp["x"].dtype, seed=R)
    y, so = gpu_scan(inp, state_in=st)
    yr, hr, Br, xr = oracle_full(inp, st)
    assert_err(to_f64(y), yr, TOL[w.dtype], "y")
    assert_err(to_f64(so.h), hr, TOL[w.dtype], "h")
    np.testing.assert_array_equal(to_f64(so.B_prev), Br)
    np.testing.assert_array_equal(to_f64(so.x_prev), xr)


def test_in_place_segmented_long_sequence():
    w = WORKLOADS["long_n128_r4"].with_(batch=1, nheads=1, seqlen=3000)
    inp = prefill_inputs(w, "cuda")
    st = random_state(1, 1, w.P, w.N, w.R, inp["x"].dtype, seed=4)
    ref = oracle_full(inp, st)
    y, _ = gpu_scan(inp, state_in=st, inplace=True)
    assert_err(to_f64(y), ref[0], TOL[w.dtype], "y")
    assert_err(to_f64(st.h), ref[1], TOL[w.dtype], "h")


def test_empty_sequence_and_empty_batch():
    w = WORKLOADS["siso_n64"].with_(batch=2, nheads=2, seqlen=0)
    inp = prefill_inputs(w, "cuda")
    st = random_state(2, 2, w.P, w.N, w.R, inp["x"].dtype, seed=5)
    y, so = gpu_scan(inp, state_in=st)
    assert y.numel() == 0
    assert torch.equal(so.h, st.h) and torch.equal(so.B_prev, st.B_prev) and torch.equal(so.x_prev, st.x_prev)
    _, so = gpu_scan(inp)          # no state in: zeros out
    assert not so.h.any() and not so.B_prev.float().any()
    w0 = WORKLOADS["siso_n64"].with_(batch=0, seqlen=16)
    inp0 = prefill_inputs(w0, "cuda")
    before = m3.launch_count()
    y0, _ = gpu_scan(inp0)
    assert y0.numel() == 0 and m3.launch_count() == before


def test_theta_pi_parity_sign_flips_on_gpu():
    """The parity mechanism (rotation by pi per 1 bit) through the CUDA path."""
    L = 64
    bits = torch.randint(0, 2, (L,), generator=torch.Generator().manual_seed(0))
    x = torch.ones(1, L, 1, 1, 4)
    B = torch.zeros(1, L, 1, 1, 2)
    C = torch.zeros(1, L, 1, 1, 2)
    C[..., 0] = 1.0
    inp = {"x": x, "B": B, "C": C, "dt": torch.ones(1, L, 1), "A": torch.zeros(1, L, 1),
           "lam": torch.ones(1, L, 1), "theta": (torch.pi * bits.float()).reshape(1, L, 1, 1)}
    inp = {k: v.cuda() for k, v in inp.items()}
    h0 = torch.zeros(1, 1, 2, 4, device="cuda")
    h0[0, 0, 0] = 1.0
    y, _ = gpu_scan(inp, state_in=m3.State(h0))
    expect = (-1.0) ** torch.cumsum(bits, 0).double()
    np.testing.assert_allclose(to_f64(y[0, :, 0, 0, 0]), expect.numpy(), atol=1e-5)


@pytest.mark.parametrize("slices", [1, 3, 7])
@pytest.mark.parametrize("groups", [0, 2])
def test_staged_host_prefill_matches_device_prefill(slices, groups):
    """mamba3_scan_fwd_staged (host buffers, copies overlapped over token ranges, the state and
    carry handed from range to range) gives the same y and final state as mamba3_scan_fwd,
    with per-head or grouped B / C."""
    w = WORKLOADS["siso_n64"].with_(batch=5, nheads=4 if groups else 3, seqlen=200)
    inp = prefill_inputs(w, "cuda")
    if groups:
        for k in ("B", "C"):
            inp[k] = _grouped(inp[k], w.nheads, groups, 2)[0]
    y_ref, s_ref = gpu_scan(inp)
    host = {k: v.cpu().pin_memory() for k, v in inp.items()}
    dev = {k: torch.empty_like(v) for k, v in inp.items()}
    y = torch.empty(inp["x"].shape, dtype=torch.float32, device="cuda")
    y_host = torch.zeros(y.shape, dtype=torch.float32).pin_memory()
    st = m3.State.zeros(w.batch, w.nheads, w.P, w.N, w.R, inp["x"].dtype)
    h_host = torch.zeros(st.h.shape, dtype=torch.float32).pin_memory()
    side = torch.cuda.Stream()
    m3.mamba3.scan_fwd_staged(host, dev, y_host, y, state_out=st, host_h=h_host, slices=slices, copy_stream=side)
    side.synchronize()
    torch.cuda.synchronize()
    assert m3.device_status() == m3.M3_OK
    tol = TOL[w.dtype]
    assert_err(y_host.double().numpy(), to_f64(y_ref), tol, "y")
    assert_err(h_host.double().numpy(), to_f64(s_ref.h), tol, "h")
    assert torch.equal(st.B_prev, s_ref.B_prev) and torch.equal(st.x_prev, s_ref.x_prev)


@pytest.mark.parametrize("wname,over,slices", [("long_n128_r4", dict(batch=1, nheads=6, seqlen=1500), 3),
                                               ("mimo_r4", dict(batch=2, nheads=5, seqlen=700), 4)])
def test_staged_host_prefill_of_segmented_ranges_matches_oracle(wname, over, slices):
    # the staged prefill from host memory where every token range is itself a segmented prefill (state
    # pass, segment pass, output pass on few sequences), the state and carry handed from range to
    # range on the device; y and the final state copied back, against the oracle
    w = WORKLOADS[wname].with_(**over)
    inp = prefill_inputs(w, "cuda")
    st_in = random_state(w.batch, w.nheads, w.P, w.N, w.R, inp["x"].dtype, seed=slices)
    host = {k: v.cpu().pin_memory() for k, v in inp.items()}
    dev = {k: torch.empty_like(v) for k, v in inp.items()}
    y = torch.empty(inp["x"].shape, dtype=torch.float32, device="cuda")
    y_host = torch.zeros(y.shape, dtype=torch.float32).pin_memory()
    st = m3.State.zeros(w.batch, w.nheads, w.P, w.N, w.R, inp["x"].dtype)
    h_host = torch.zeros(st.h.shape, dtype=torch.float32).pin_memory()
    side = torch.cuda.Stream()
    m3.mamba3.scan_fwd_staged(host, dev, y_host, y, state_in=st_in, state_out=st, host_h=h_host, slices=slices,
                              copy_stream=side)
    side.synchronize()
    torch.cuda.synchronize()
    assert m3.device_status() == m3.M3_OK
    yr, hr, Br, xr = oracle_full(inp, st_in)
    tol = TOL[w.dtype]
    assert_err(y_host.double().numpy(), yr, tol, "y")
    assert_err(h_host.double().numpy(), hr, tol, "h")
    np.testing.assert_array_equal(to_f64(st.B_prev), Br)
    np.testing.assert_array_equal(to_f64(st.x_prev), xr)


# ---------------------------------------------------------------- output element type

Y16 = (torch.float16, torch.bfloat16)


@pytest.mark.parametrize("case", ["siso_n64_small", "mimo_r4_small", "long_small_segmented", "siso_n128_small",
                                  "siso_n64_small_f32", "odd_shapes_bf16"])
def test_prefill_16bit_y_is_the_fp32_result_rounded_once(case):
    # the same arithmetic for every output type: y in fp16 / bf16 equals the fp32 y rounded to
    # nearest even, bit for bit (tensor-core and SIMT paths)
    wname, over = SMALL[case]
    w = WORKLOADS[wname].with_(**over)
    inp = prefill_inputs(w, "cuda")
    st = random_state(w.batch, w.nheads, w.P, w.N, w.R, inp["x"].dtype, seed=3)
    y32 = m3.scan_fwd(*(inp[k] for k in KEYS), state_in=st)
    for yd in Y16:
        y = m3.scan_fwd(*(inp[k] for k in KEYS), state_in=st, y_dtype=yd)
        assert y.dtype == yd
        assert torch.equal(y, y32.to(yd)), yd
    assert m3.device_status() == m3.M3_OK


@pytest.mark.parametrize("wname", ["siso_n64", "siso_n128", "mimo_r4"])
def test_prefill_fp16_y_full_size_sampled_matches_oracle(wname):
    # fp16 y keeps y at the input element size; rounding costs at most 2^-11 |y|, inside the bar
    w = WORKLOADS[wname]
    inp = prefill_inputs(w, "cuda")
    so = m3.State.zeros(w.batch, w.nheads, w.P, w.N, w.R, inp["x"].dtype)
    y = m3.scan_fwd(*(inp[k] for k in KEYS), state_out=so, y_dtype=torch.float16)
    assert m3.device_status() == m3.M3_OK
    pairs = [(0, 0), (w.batch // 2, w.nheads // 3), (w.batch - 1, w.nheads - 1)]
    stack = {k: torch.cat([inp[k][b:b + 1, :, h:h + 1] for b, h in pairs], dim=0) for k in KEYS}
    yr, hr, _, _ = oracle.scan(*(to_f64(stack[k]) for k in KEYS), nthreads=len(pairs))
    for i, (b, h) in enumerate(pairs):
        assert_err(to_f64(y[b:b + 1, :, h:h + 1]), yr[i:i + 1], TOL[w.dtype], f"y (b, h) = {(b, h)}")
        assert_err(to_f64(so.h[b:b + 1, h:h + 1]), hr[i:i + 1], TOL[w.dtype], f"h (b, h) = {(b, h)}")
    assert torch.isfinite(y.float()).all()


@pytest.mark.parametrize("over", [dict(), dict(dtype="f32"), dict(P=16, dtype="f32")])
def test_decode_16bit_y_is_the_fp32_result_rounded_once(over):
    # tensor-core, streaming and generic decode kernels
    w = WORKLOADS["decode_n64_r4"].with_(batch=3, nheads=6, **over)
    st = decode_state(w, "cuda")
    tok = decode_pool(w, "cuda", pool=1)[0]
    s32 = m3.State(st["h"].clone(), st["B_prev"].clone(), st["x_prev"].clone())
    y32 = m3.decode_step(*(tok[k] for k in KEYS), state=s32)
    for yd in Y16:
        s = m3.State(st["h"].clone(), st["B_prev"].clone(), st["x_prev"].clone())
        y = m3.decode_step(*(tok[k] for k in KEYS), state=s, y_dtype=yd)
        assert y.dtype == yd
        assert torch.equal(y, y32.to(yd)), yd
        assert torch.equal(s.h, s32.h)


# ---------------------------------------------------------------- the chunk rule Q = N / R

@pytest.mark.parametrize("R,H,b,L,with_state", [(1, 3, 2, 300, False), (2, 2, 1, 333, True), (4, 3, 1, 201, True),
                                                (4, 2, 1, 3000, False), (1, 1, 1, 5000, True)])
def test_chunk_rule_tile_matches_oracle(R, H, b, L, with_state):
    # dims.chunk = N / R selects the 64-row tile for N = 64 (linkstar.cloud/article/869, section
    # "训练怎么办"); long sequences with few heads are also cut into segments
    w = WORKLOADS["mimo_r4"].with_(batch=b, nheads=H, seqlen=L, R=R)
    inp = prefill_inputs(w, "cuda")
    st = random_state(b, H, w.P, w.N, R, inp["x"].dtype, seed=R) if with_state else None
    y, so = gpu_scan(inp, state_in=st, chunk=64 // R)
    yr, hr, Br, xr = oracle_full(inp, st)
    assert_err(to_f64(y), yr, TOL[w.dtype], "y")
    assert_err(to_f64(so.h), hr, TOL[w.dtype], "h")
    np.testing.assert_array_equal(to_f64(so.B_prev), Br)
    # and it agrees with the default tile
    y0, _ = gpu_scan(inp, state_in=st)
    assert_err(to_f64(y), to_f64(y0), TOL[w.dtype], "y tiles")


def test_chunk_rule_tile_with_bc_matches_oracle():
    w = WORKLOADS["mimo_r4"].with_(batch=1, nheads=2, seqlen=2500)
    inp = prefill_inputs(w, "cuda")
    from selective_state_space_134_b300.synth import bc_params
    p = bc_params(w, "cuda", seed=7)
    bc = m3.BcNorm(p["B_weight"], p["B_bias"], p["C_weight"], p["C_bias"], p["eps"])
    y = m3.scan_fwd(*(inp[k] for k in KEYS), chunk=16, bc=bc)
    assert m3.device_status() == m3.M3_OK
    bref = {k: (to_f64(v) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
    yr, _, _, _ = oracle.scan_bc(*(to_f64(inp[k]) for k in KEYS), bref, nthreads=2)
    assert_err(to_f64(y), yr, TOL[w.dtype], "y")


# ---------------------------------------------------------------- failure detection

def test_bounded_wait_reports_timeout_and_the_context_stays_usable():
    # a kernel waits on a barrier nothing completes; the bounded wait gives up after 1 ms and the
    # timeout reaches the host through the device status word, once; then a prefill still runs right
    from selective_state_space_134_b300 import mamba3 as api
    assert m3.device_status() == m3.M3_OK
    assert m3.lib().mamba3_selftest_wait_timeout(1_000_000, None) == api.M3_OK
    assert m3.device_status() == api.M3_ERR_TIMEOUT
    assert m3.device_status() == m3.M3_OK            # read and cleared
    assert m3.lib().mamba3_selftest_wait_timeout(0, None) == api.M3_ERR_INVALID_ARG
    w = WORKLOADS["siso_n64"].with_(batch=1, nheads=2, seqlen=150)
    inp = prefill_inputs(w, "cuda")
    y, so = gpu_scan(inp)
    yr, hr, _, _ = oracle_full(inp)
    assert_err(to_f64(y), yr, TOL[w.dtype], "y")


# ---------------------------------------------------------------- more sequences than SMs (several waves of CTAs)

@pytest.mark.parametrize("N,R,b,H,L,with_state,kw", [
    (64, 4, 3, 60, 300, False, {}), (64, 4, 2, 90, 257, True, {}), (128, 1, 1, 200, 333, True, {}),
    (64, 1, 4, 50, 650, False, dict(y_dtype=torch.float16)), (64, 2, 2, 100, 200, True, dict(chunk=32)),
    (128, 4, 1, 170, 97, False, {})])
def test_more_sequences_than_sms_match_oracle(N, R, b, H, L, with_state, kw):
    # b x H > SMs: several waves of one-sequence CTAs, with a carry, fp16 y and the chunk rule
    w = WORKLOADS["mimo_r4"].with_(batch=b, nheads=H, seqlen=L, N=N, R=R)
    inp = prefill_inputs(w, "cuda")
    st = random_state(b, H, w.P, N, R, inp["x"].dtype, seed=11) if with_state else None
    so = m3.State.zeros(b, H, w.P, N, R, inp["x"].dtype)
    y = m3.scan_fwd(*(inp[k] for k in KEYS), state_in=st, state_out=so, **kw)
    assert m3.device_status() == m3.M3_OK
    yr, hr, Br, xr = oracle_full(inp, st)
    assert_err(to_f64(y), yr, TOL[w.dtype], "y")
    assert_err(to_f64(so.h), hr, TOL[w.dtype], "h")
    np.testing.assert_array_equal(to_f64(so.B_prev), Br)
    np.testing.assert_array_equal(to_f64(so.x_prev), xr)
    # twice in a row: the same result
    y2 = m3.scan_fwd(*(inp[k] for k in KEYS), state_in=st, **kw)
    assert torch.equal(y, y2)


@pytest.mark.parametrize("N,R,b,H,G,L", [(64, 4, 4, 40, 8, 300), (64, 1, 5, 36, 12, 333), (128, 4, 2, 80, 20, 150)])
def test_more_sequences_than_sms_with_grouped_bc_match_oracle(N, R, b, H, G, L):
    # more sequences than SMs (the balanced pass: equal chunk ranges over one CTA per SM, its own input
    # maps) with B and C shared by groups of H / G heads, an initial state and a carry; against the
    # oracle on the per-head expansion
    w = WORKLOADS["mimo_r4"].with_(batch=b, nheads=H, seqlen=L, N=N, R=R)
    inp = prefill_inputs(w, "cuda")
    full = dict(inp)
    for k in ("B", "C"):
        inp[k], full[k] = _grouped(inp[k], H, G, 2)
    st = random_state(b, H, w.P, N, R, inp["x"].dtype, seed=G)
    y, so = gpu_scan(inp, state_in=st)
    yr, hr, Br, xr = oracle_full(full, st)
    assert_err(to_f64(y), yr, TOL[w.dtype], "y")
    assert_err(to_f64(so.h), hr, TOL[w.dtype], "h")
    np.testing.assert_array_equal(to_f64(so.B_prev), Br)
    np.testing.assert_array_equal(to_f64(so.x_prev), xr)


def test_more_sequences_than_sms_with_bc_match_oracle():
    from selective_state_space_134_b300.synth import bc_params
    w = WORKLOADS["mimo_r4"].with_(batch=2, nheads=96, seqlen=180)
    inp = prefill_inputs(w, "cuda")
    p = bc_params(w, "cuda", seed=5)
    bc = m3.BcNorm(p["B_weight"], p["B_bias"], p["C_weight"], p["C_bias"], p["eps"])
    y = m3.scan_fwd(*(inp[k] for k in KEYS), bc=bc)
    assert m3.device_status() == m3.M3_OK
    bref = {k: (to_f64(v) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
    yr, _, _, _ = oracle.scan_bc(*(to_f64(inp[k]) for k in KEYS), bref, nthreads=8)
    assert_err(to_f64(y), yr, TOL[w.dtype], "y")
