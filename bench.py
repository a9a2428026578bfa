"""Benchmark of the Mamba-3 layer recurrence on B300: prefill and decode tokens/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--quick] [--decode-only]
    python bench.py --workload NAME [--batch B] [--heads H] [--seqlen L] [--backward] [--steps K]

A step is one mamba3_scan_fwd over the SISO bf16 prefill workload (batch 4,
32 heads, L = 4096, P = 64, N = 64, R = 1): the prefill hot path end to end
(prefix + RoPE, in-chunk contraction, state passing, outputs and final
state).  `value` = prefill tokens/s (batch x L / time; a token covers every
head), inputs resident in HBM and larger than L2 (no flush needed).  The same
line carries the decode-step measurement (batch 256, 32 heads, one token per
call over 1024 calls; also N = 64, R = 4 on a 512-slot state pool), the other
prefill workloads (N = 128, MIMO R = 4, long context, and the headline shape
with grouped B / C), the roofline of the dominant kernel (timed live by CUDA
events around all timed steps on the launch stream, so rates are per step,
gaps included: the library launches its kernels as programmatic dependents of
the kernel before them, and trace events between launches would serialise
them; a step of several launches also reports the output pass's own time from
a second, traced run; `traffic` from profiles/traffic.json while the library
sources match its digest), the end-to-end figure through host
buffers, the clocks seen, and the fp64 CPU oracle timed on this host's cores.
--quick prints the headline alone; --decode-only prints the decode workloads
alone.

--impl reference times the CPU oracle itself on the same workload (the
reference arm of this method: there is no GPU implementation to compare with).
Under torchrun every rank runs an independent replica on its own GPU (the
sequences are independent: weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

HEADLINE = "siso_n64"
KEYS = ("x", "B", "C", "dt", "A", "lam", "theta")


def bytes_per_token_head(w, groups=0) -> float:
    """Algorithmic HBM bytes of prefill per (token, head), every tensor at the input element
    size e: e (2PR + 2NR + N/2 + 3) for x and y; B and C (shared by nheads / groups heads when
    grouped); theta; dt, A, lambda."""
    e = 4 if w.dtype == "f32" else 2
    share = groups / w.nheads if groups else 1.0
    return e * (2 * w.P * w.R + 2 * w.N * w.R * share + w.N // 2 + 3)


def y_surplus_per_token_head(w, y_bytes=4) -> float:
    """Bytes per (token, head) that a y wider than the input element (fp32 y for bf16 inputs)
    moves beyond the algorithmic count; reported beside the roofline, never folded into it."""
    e = 4 if w.dtype == "f32" else 2
    return max(0, y_bytes - e) * w.P * w.R


def prefill_bytes(w, groups=0) -> int:
    """Whole prefill step: every (token, head), plus the final state (fp32) and carry written."""
    bh = w.batch * w.nheads
    return int(w.token_heads * bytes_per_token_head(w, groups)) + bh * w.N * w.P * 4 + \
        bh * w.R * (w.N + w.P) * (4 if w.dtype == "f32" else 2)


def decode_bytes(w) -> int:
    """Per call: state read + write (fp32), carry read + write, token inputs and y at the input
    element size."""
    e = 4 if w.dtype == "f32" else 2
    bh = w.batch * w.nheads
    return bh * (8 * w.N * w.P + 2 * e * w.R * (w.N + w.P) + e * (2 * w.R * w.N + w.R * w.P + w.N // 2 + 3)
                 + e * w.R * w.P)


def decode_y_surplus(w, y_bytes=4) -> int:
    e = 4 if w.dtype == "f32" else 2
    return w.batch * w.nheads * max(0, y_bytes - e) * w.R * w.P


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6400.0, 1800.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (every 50 ms) around a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            ident = str(device_index)
        self.ident = ident

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.ident, f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
                except Exception:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if self.t0 is not None and self.t0 - 1 <= r[0] <= self.t1 + 1] or rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for n, v in zip(names, r[3]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median([r[1] for r in inside]) if inside else None,
                "sm_max_mhz": max([r[2] for r in inside]) if inside else None,
                "reasons": sorted(reasons), "samples": len(inside)}


# ------------------------------------------------------------------ distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    if ws <= 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ our arm
def time_prefill(m3, w, steps, warmup, trace_kernel=None, groups=0, y_dtype=torch.float32, bc=False, chunk=0):
    """Device time of `steps` scan_fwd calls (inputs resident). Returns dict.  groups > 0: B and C
    shared by groups of nheads / groups heads (the first head's values of each group); y_dtype:
    element type of y; bc: with BC normalisation and bias (synthetic gains and biases); chunk: tokens
    per chunk (0: the library's tile)."""
    from selective_state_space_134_b300.synth import prefill_inputs
    inp = prefill_inputs(w, "cuda")
    if groups:
        idx = torch.arange(0, w.nheads, w.nheads // groups, device="cuda")
        for k in ("B", "C"):
            inp[k] = inp[k].index_select(2, idx).contiguous()
    dtype = inp["x"].dtype
    st = m3.State.zeros(w.batch, w.nheads, w.P, w.N, w.R, dtype)
    y = torch.empty(inp["x"].shape, dtype=y_dtype, device="cuda")
    ws_bytes = m3.scan_fwd_workspace(m3.dims(w.batch, w.seqlen, w.nheads, w.P, w.N, w.R, dtype, chunk=chunk,
                                             ngroups=groups if groups != w.nheads else 0))
    work = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    args = [inp[k] for k in KEYS]
    bcn = None
    if bc:
        from selective_state_space_134_b300.synth import bc_params
        p = bc_params(w, "cuda")
        bcn = m3.BcNorm(p["B_weight"], p["B_bias"], p["C_weight"], p["C_bias"], p["eps"])

    def step():
        m3.scan_fwd(*args, state_out=st, y=y, workspace=work, bc=bcn, chunk=chunk)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    n0 = m3.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    launches = m3.launch_count() - n0
    ms = e0.elapsed_time(e1)
    traced = (0, 0.0)
    if trace_kernel is not None and launches > steps:
        # several launches a step: the traced kernel's own time from a second run of the same steps
        # (trace events between launches would hold back the programmatic dependent launches of the
        # timed run, so they stay out of it)
        m3.trace_begin(trace_kernel, steps)
        for _ in range(steps):
            step()
        torch.cuda.synchronize()
        traced = m3.trace_end()
    assert m3.device_status() == m3.M3_OK
    return {"ms": ms, "launches": launches, "traced": traced, "inputs": inp, "ws": ws_bytes}


def prefill_line(m3, w, res, steps, hbm_peak, peak_kind, groups=0, y_bytes=4):
    """Tokens/s and the HBM roofline of one prefill workload.  `frac` covers the whole step (all
    launches): algorithmic bytes / time per step.  The output pass's own rate (the same bytes over
    its traced time) is reported beside it; for one-launch steps the two agree."""
    ms_step = res["ms"] / steps
    n_tr, tr_ms = res["traced"]
    algo = prefill_bytes(w, groups)
    k_ms = tr_ms / n_tr if n_tr else ms_step
    achieved = algo / (ms_step * 1e-3) / 1e9
    achieved_k = algo / (k_ms * 1e-3) / 1e9
    return {
        "tokens_per_s": w.batch * w.seqlen / (ms_step * 1e-3),
        "ms_per_step": ms_step,
        "roofline": {"bound": "hbm", "kernel": "whole prefill step", "achieved": round(achieved, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "traffic": (traffic_for("prefill_output", w.name + (f"_g{groups}" if groups else ""))
                                 if _full_size(w) else None),
                     "algorithmic_bytes": algo,
                     "extra_bytes_wide_y": int(w.token_heads * y_surplus_per_token_head(w, y_bytes)),
                     "y_bytes": y_bytes,
                     "output_pass": {"kernel_ms": k_ms, "achieved": round(achieved_k, 1),
                                     "frac": round(achieved_k / hbm_peak, 4)},
                     "peak_source": peak_kind},
    }


def _full_size(w) -> bool:
    """The traffic records are of the named workloads at their own sizes: a resized run has none."""
    from selective_state_space_134_b300.synth import WORKLOADS
    ref = WORKLOADS.get(w.name)
    return ref is not None and ref.token_heads == w.token_heads and ref.R == w.R and ref.N == w.N


def traffic_for(kernel, workload):
    """ncu DRAM bytes per launch recorded under profiles/ for the current sources of that kernel, else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        from selective_state_space_134_b300.build import source_digest
        r = rec.get(f"{kernel}/{workload}")
        if r and r.get("source_digest") == source_digest(kernel):
            return r["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


def time_decode(m3, w, calls, warmup):
    from selective_state_space_134_b300.synth import decode_pool, decode_state
    st = decode_state(w, "cuda")
    state = m3.State(st["h"], st["B_prev"], st["x_prev"])
    pool = decode_pool(w, "cuda")
    ys = [torch.empty(p["x"].shape, dtype=torch.float32, device="cuda") for p in pool]
    argsets = [[p[k] for k in KEYS] for p in pool]
    for i in range(warmup):
        m3.decode_step(*argsets[i % len(pool)], state=state, y=ys[i % len(pool)])
    torch.cuda.synchronize()
    # no per-launch trace events here: consecutive steps are programmatic dependents of one another,
    # and an event between two launches would serialise them; the kernel time is the per-call time
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(calls):
        m3.decode_step(*argsets[i % len(pool)], state=state, y=ys[i % len(pool)])
    e1.record()
    torch.cuda.synchronize()
    assert m3.device_status() == m3.M3_OK
    ms = e0.elapsed_time(e1) / calls
    return ms, ms


def time_decode_pooled(m3, w, calls, warmup, pool_factor=2):
    """The decode step on states kept in a pool of pool_factor x batch slots: the batch rows name a
    seeded random set of distinct slots (serving with a state pool)."""
    from selective_state_space_134_b300.synth import decode_pool, decode_state
    S = pool_factor * w.batch
    ps = decode_state(w.with_(batch=S), "cuda")
    pool = m3.State(ps["h"], ps["B_prev"], ps["x_prev"])
    g = torch.Generator().manual_seed(1234)
    slot = torch.randperm(S, generator=g)[: w.batch].to(torch.int32).to("cuda")
    toks = decode_pool(w, "cuda")
    ys = [torch.empty(p["x"].shape, dtype=torch.float32, device="cuda") for p in toks]
    argsets = [[p[k] for k in KEYS] for p in toks]
    for i in range(warmup):
        m3.decode_step_pooled(*argsets[i % len(toks)], slot=slot, pool=pool, y=ys[i % len(toks)])
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(calls):
        m3.decode_step_pooled(*argsets[i % len(toks)], slot=slot, pool=pool, y=ys[i % len(toks)])
    e1.record()
    torch.cuda.synchronize()
    assert m3.device_status() == m3.M3_OK
    ms = e0.elapsed_time(e1) / calls
    return ms, ms


def e2e_prefill(m3, w, inp, steps, warmup, slices=8):
    """Same metric through host buffers, via the library's staged prefill: every step copies the
    inputs in from pinned host memory and y and the final state h back out, the copies of each
    token range overlapped with the kernels and copies of the others."""
    host = {k: v.cpu().pin_memory() for k, v in inp.items()}
    dtype = inp["x"].dtype
    dev = {k: torch.empty_like(v) for k, v in inp.items()}
    st = m3.State.zeros(w.batch, w.nheads, w.P, w.N, w.R, dtype)
    y = torch.empty(inp["x"].shape, dtype=torch.float32, device="cuda")
    y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    h_host = torch.empty(st.h.shape, dtype=st.h.dtype).pin_memory()
    slices = max(1, min(slices, w.seqlen))
    need = m3.mamba3.scan_fwd_staged_workspace(m3.dims(w.batch, w.seqlen, w.nheads, w.P, w.N, w.R, dtype), slices)
    work = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    main, side = torch.cuda.current_stream(), torch.cuda.Stream()

    def step():
        m3.mamba3.scan_fwd_staged(host, dev, y_host, y, state_out=st, host_h=h_host, slices=slices,
                                  workspace=work, stream=main, copy_stream=side)

    for _ in range(warmup):
        step()
    main.wait_stream(side)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for _ in range(steps):
        step()
    main.wait_stream(side)
    e1.record(main)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = y.numel() * y.element_size() + st.h.numel() * 4
    return {"value": w.batch * w.seqlen / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "api": "mamba3_scan_fwd_staged",
            "slices": slices}


def _oracle_sample(w, nseq, max_tokens=None):
    """CPU inputs for `nseq` (b, h) sequences of workload w (heads stacked as the batch axis) of at most
    `max_tokens` tokens each, widened to float64 for the oracle (same distributions as the GPU runs)."""
    from selective_state_space_134_b300.synth import prefill_inputs, to_f64
    L = w.seqlen if max_tokens is None else min(w.seqlen, max_tokens)
    inp = prefill_inputs(w.with_(batch=nseq, nheads=1, seqlen=max(L, 1)), "cpu")
    return [to_f64(inp[k]) for k in KEYS], L


def oracle_rate(w, threads, seconds, max_tokens=None, nseq=None):
    """Times the fp64 CPU oracle on a bounded sample of workload w: `nseq` whole (b, h) sequences
    (default 2 x threads) of at most `max_tokens` tokens, scanned again and again for about `seconds`
    of wall time on `threads` POSIX threads.  Returns tokens/s, a token counting all the workload's
    heads (the GPU figures count the same way)."""
    import oracle
    nseq = nseq or max(1, min(w.batch * w.nheads, 2 * threads))
    arrs, L = _oracle_sample(w, nseq, max_tokens)
    reps, t = 0, time.perf_counter()
    while True:
        oracle.scan(*arrs, nthreads=threads)
        reps += 1
        sec = time.perf_counter() - t
        if sec >= seconds:
            break
    return {"value": reps * nseq * L / w.nheads / sec, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{nseq} of {w.batch * w.nheads} (b,h) sequences x {L} of {w.seqlen} tokens of {w.name}, "
                      f"scanned {reps} times ({sec:.1f} s); a token counts all {w.nheads} heads",
            "seconds": round(sec, 2)}


def oracle_decode_rate(w, threads, seconds):
    """The oracle's decode step (the recurrence with L = 1) on a sample of 64 x threads (b, h) rows."""
    import oracle
    from selective_state_space_134_b300.synth import decode_pool, decode_state, to_f64
    rows = min(w.batch * w.nheads, 64 * threads)
    ws = w.with_(batch=rows, nheads=1)
    st = decode_state(ws, "cpu")
    tok = decode_pool(ws, "cpu", pool=1)[0]
    args = [to_f64(tok[k]) for k in KEYS] + [to_f64(st["h"]), to_f64(st["B_prev"]), to_f64(st["x_prev"])]
    reps, t = 0, time.perf_counter()
    while True:
        x, B, C, dt, A, lam, th, h, Bp, xp = args
        oracle.scan(x[:, None], B[:, None], C[:, None], dt[:, None], A[:, None], lam[:, None], th[:, None],
                    h0=h, Bprev=Bp, xprev=xp, nthreads=threads)
        reps += 1
        sec = time.perf_counter() - t
        if sec >= seconds:
            break
    # decode tokens/s: one token per batch row, all heads
    return {"value": reps * rows / w.nheads / sec, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} of {w.batch * w.nheads} (b,h) rows, one step, {reps} times ({sec:.1f} s)",
            "seconds": round(sec, 2)}


def cpu_baseline_table(seconds=1.5):
    """The oracle per workload, single-thread and on every host core (the long-context workload on
    its first 4096 tokens of 2 x cores sequences)."""
    from selective_state_space_134_b300.synth import WORKLOADS
    cores = os.cpu_count() or 1
    out = {}
    for name in ("tiny_f32", "siso_n64", "siso_n128", "mimo_r4", "long_n128_r4"):
        w = WORKLOADS[name]
        cap = 4096 if name == "long_n128_r4" else None
        one = oracle_rate(w, 1, seconds, cap, nseq=1)
        allc = oracle_rate(w, cores, seconds, cap)
        out[name] = {"single_thread": round(one["value"], 1), "all_cores": round(allc["value"], 1),
                     "cores": cores, "sample_all_cores": allc["sample"]}
    for name in ("decode_n64_r1", "decode_n64_r4", "decode_n128_r1", "decode_n128_r4"):
        w = WORKLOADS[name]
        one = oracle_decode_rate(w, 1, seconds / 2)
        allc = oracle_decode_rate(w, cores, seconds / 2)
        out[name] = {"single_thread": round(one["value"], 1), "all_cores": round(allc["value"], 1),
                     "cores": cores, "sample_all_cores": allc["sample"]}
    return out


def time_backward(m3, w, steps, warmup):
    """Device time of `steps` mamba3_scan_bwd calls on workload w (dy ~ N(0, 1), inputs resident)."""
    from selective_state_space_134_b300.synth import prefill_inputs
    inp = prefill_inputs(w, "cuda")
    g = torch.Generator(device="cuda").manual_seed(5)
    dy = torch.randn(inp["x"].shape, device="cuda", generator=g)
    args = [inp[k] for k in KEYS]
    d = m3.dims(w.batch, w.seqlen, w.nheads, w.P, w.N, w.R, inp["x"].dtype)
    work = torch.empty(max(m3.scan_bwd_workspace(d), 1), dtype=torch.uint8, device="cuda")
    grads = m3.scan_bwd(*args, dy, workspace=work)
    for _ in range(warmup):
        m3.scan_bwd(*args, dy, workspace=work, grads=grads)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        m3.scan_bwd(*args, dy, workspace=work, grads=grads)
    e1.record()
    torch.cuda.synchronize()
    assert m3.device_status() == m3.M3_OK
    return e0.elapsed_time(e1) / steps, work.numel()


def backward_flops(w):
    """fp32 flops of the backward kernel (its contractions; 2 per FMA).  Per chunk of QR rows (t, r):
    S and Z (causal halves, QR^2 (N + P) / 2), dX's score term (QR^2 P / 2), dB~'s and dC~'s score terms
    (QR^2 N), and five N x P x QR products (checkpoint update, B~ D~, dY H'^T, X D~^T, state gradient)."""
    rows = 16 if w.N * w.P > 4096 else 32
    Q = max(1, rows // w.R)
    QR = Q * w.R
    fma = QR * QR * (w.N + w.P) / 2 + QR * QR * w.P / 2 + QR * QR * w.N + 5 * QR * w.N * w.P
    return 2.0 * fma / Q * w.token_heads


def fp32_peak_tflops():
    """fp32 CUDA-core peak: SMs x 128 lanes x 2 flops (FMA) x the maximum SM clock."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", 2032.0))
    except Exception:
        mhz = 2032.0
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return sms * 128 * 2 * mhz * 1e6 / 1e12


def run_ours(args):
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(ws, "nccl")
    import selective_state_space_134_b300 as m3
    from selective_state_space_134_b300.synth import WORKLOADS
    m3.lib()
    hbm_peak, _, peak_kind = peaks()
    w = WORKLOADS[HEADLINE]

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    # headline: warm-up + timed region, barrier + synchronize on both sides
    from selective_state_space_134_b300.synth import prefill_inputs
    inp = prefill_inputs(w, "cuda")
    dtype = inp["x"].dtype
    st = m3.State.zeros(w.batch, w.nheads, w.P, w.N, w.R, dtype)
    y = torch.empty(inp["x"].shape, dtype=torch.float32, device="cuda")
    ws_bytes = m3.scan_fwd_workspace(m3.dims(w.batch, w.seqlen, w.nheads, w.P, w.N, w.R, dtype))
    work = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    a = [inp[k] for k in KEYS]
    for _ in range(args.warmup):
        m3.scan_fwd(*a, state_out=st, y=y, workspace=work)
    barrier(ws)
    torch.cuda.synchronize()
    # one launch a step: the step's CUDA-event time is the kernel's (no per-launch trace events in the
    # timed region; they would hold back the programmatic dependent launches)
    n0 = m3.launch_count()
    if sampler:
        sampler.mark("t0")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        m3.scan_fwd(*a, state_out=st, y=y, workspace=work)
    e1.record()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t1")
    barrier(ws)
    launches = m3.launch_count() - n0
    ms = max_over_ranks(e0.elapsed_time(e1), ws)
    traced = (0, 0.0)
    status = m3.device_status()
    clocks = sampler.stop() if sampler else None
    if status != m3.M3_OK:
        raise RuntimeError(f"device status {m3.status_string(status)}")
    head = prefill_line(m3, w, {"ms": ms, "traced": traced}, args.steps, hbm_peak, peak_kind)
    ms_step = ms / args.steps
    value = ws * w.batch * w.seqlen / (ms_step * 1e-3)

    extra = {}
    if rank == 0 and not args.quick:
        # decode: the four (N, R) variants, 1024 calls each
        dec = decode_results(m3, hbm_peak)
        extra["decode"] = {"metric": "decode tokens/s", "unit": "tokens/s", "workloads": dec}
        # other prefill workloads
        pre = {}
        # (at least 3 warm-up steps, and enough timed steps that host-side call overhead and the
        # queue's start stay out of the rate: tens of milliseconds a workload)
        for name, steps in (("siso_n128", 100), ("mimo_r4", 10), ("long_n128_r4", 3)):
            wp = WORKLOADS[name]
            r = time_prefill(m3, wp, steps, 3, m3.KERNEL_PREFILL_OUTPUT)
            pre[name] = prefill_line(m3, wp, r, steps, hbm_peak, peak_kind)
            pre[name]["launches_per_step"] = r["launches"] / steps
            del r
            torch.cuda.empty_cache()
        # variants of the headline shape (and of MIMO): grouped B / C (one B and C per 8 heads), fp16 y,
        # BC normalisation and bias, and the chunk rule Q = N / R of the pages
        wp = WORKLOADS[HEADLINE]
        variants = (("siso_n64_grouped_g4", HEADLINE, dict(groups=4)),
                    ("siso_n64_y_f16", HEADLINE, dict(y_dtype=torch.float16)),
                    ("siso_n64_bc", HEADLINE, dict(bc=True)),
                    ("siso_n64_chunk_rule_q64", HEADLINE, dict(chunk=64)),
                    ("mimo_r4_bc", "mimo_r4", dict(bc=True)),
                    ("mimo_r4_chunk_rule_q16", "mimo_r4", dict(chunk=16)))
        for key, name, kw in variants:
            wp = WORKLOADS[name]
            steps = 100 if name == HEADLINE else 10
            r = time_prefill(m3, wp, steps, 3, m3.KERNEL_PREFILL_OUTPUT, **kw)
            pre[key] = prefill_line(m3, wp, r, steps, hbm_peak, peak_kind, groups=kw.get("groups", 0),
                                    y_bytes=kw.get("y_dtype", torch.float32).itemsize)
            pre[key]["launches_per_step"] = r["launches"] / steps
            del r
            torch.cuda.empty_cache()
        extra["prefill"] = pre
        # backward pass (training): siso_n64 and mimo_r4; the ALU roofline of its fp32 contractions
        bwd = {}
        for name, steps in ((HEADLINE, 5), ("mimo_r4", 2)):
            wb = WORKLOADS[name]
            ms_b, ws_b = time_backward(m3, wb, steps, 3)
            fl = backward_flops(wb)
            peak = fp32_peak_tflops()
            bwd[name] = {"tokens_per_s": wb.batch * wb.seqlen / (ms_b * 1e-3), "ms_per_step": ms_b,
                         "workspace_bytes": ws_b,
                         "roofline": {"bound": "alu", "achieved": round(fl / (ms_b * 1e-3) / 1e12, 3),
                                      "peak": round(peak, 1), "unit": "TFLOP/s",
                                      "frac": round(fl / (ms_b * 1e-3) / 1e12 / peak, 4),
                                      "flops": fl, "peak_source": "derived: SMs x 128 fp32 lanes x 2 x max clock"}}
            torch.cuda.empty_cache()
        extra["backward"] = {"metric": "backward tokens/s", "unit": "tokens/s", "workloads": bwd}

    e2e = e2e_prefill(m3, w, inp, max(2, min(args.steps, 10)), 3) if rank == 0 else None
    cpu = None
    if rank == 0 and ws == 1 and not args.quick:
        cpu = oracle_rate(w, os.cpu_count() or 1, 10.0)
        cpu["per_workload"] = cpu_baseline_table()

    if rank == 0:
        line = {
            "metric": "prefill tokens/s", "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{HEADLINE}: SISO bf16 prefill, batch {w.batch}, heads {w.nheads}, "
                                   f"L={w.seqlen}, P={w.P}, N={w.N}, R={w.R}",
                       "batch": w.batch, "heads": w.nheads, "seq_len": w.seqlen, "P": w.P, "N": w.N, "R": w.R,
                       "l2": f"inputs larger than L2 ({prefill_bytes(w) / 1e6:.0f} MB per step), no flush",
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
            "roofline": head["roofline"],
            "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
        }
        if cpu:
            line["cpu_baseline"] = cpu
        line.update(extra)
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ reference arm (the CPU oracle)
def run_reference(args):
    """The reference arm: the fp64 CPU oracle on this host's cores, on the headline workload, timed
    with the same sampling as the bench line's cpu_baseline; each step a bounded sample."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from selective_state_space_134_b300.synth import WORKLOADS
    w = WORKLOADS[HEADLINE]
    cores = os.cpu_count() or 1
    oracle_rate(w, cores, 0.5)                       # warm-up (input generation, library load)
    per_step = max(1.0, min(10.0, 120.0 / max(args.steps, 1)))
    r = oracle_rate(w, cores, per_step * args.steps)
    value = r["value"]
    sec = args.steps and r["seconds"] / args.steps
    print(json.dumps({
        "impl": "reference", "metric": "prefill tokens/s", "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{HEADLINE}: SISO bf16 prefill, batch {w.batch}, heads {w.nheads}, "
                               f"L={w.seqlen}, P={w.P}, N={w.N}, R={w.R}"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": r["sample"]},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def decode_results(m3, hbm_peak, calls=1024, warmup=16):
    """The four decode workloads (and N=64 R=4 on a state pool): tokens/s, us per call and the
    kernel's HBM roofline."""
    from selective_state_space_134_b300.synth import WORKLOADS
    dec = {}
    for name in ("decode_n64_r1", "decode_n64_r4", "decode_n128_r1", "decode_n128_r4"):
        wd = WORKLOADS[name]
        ms_call, k_ms = time_decode(m3, wd, calls, warmup)
        gbs = decode_bytes(wd) / (k_ms * 1e-3) / 1e9
        dec[name] = {"tokens_per_s": wd.batch / (ms_call * 1e-3), "us_per_call": round(ms_call * 1e3, 2),
                     "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                                  "frac": round(gbs / hbm_peak, 4),
                                  "traffic": traffic_for("decode", name),
                                  "algorithmic_bytes": decode_bytes(wd), "kernel_ms": k_ms,
                                  "extra_bytes_wide_y": decode_y_surplus(wd)}}
    # the same step on a state pool (2 x batch slots, rows on a random set of distinct slots)
    wd = WORKLOADS["decode_n64_r4"]
    ms_call, k_ms = time_decode_pooled(m3, wd, calls, warmup)
    gbs = decode_bytes(wd) / (k_ms * 1e-3) / 1e9
    dec["decode_n64_r4_pooled"] = {
        "tokens_per_s": wd.batch / (ms_call * 1e-3), "us_per_call": round(ms_call * 1e3, 2),
        "pool_slots": 2 * wd.batch,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(gbs / hbm_peak, 4), "traffic": traffic_for("decode", "decode_n64_r4_pooled"),
                     "algorithmic_bytes": decode_bytes(wd), "kernel_ms": k_ms,
                     "extra_bytes_wide_y": decode_y_surplus(wd)}}
    return dec


def run_decode_only(args):
    torch.cuda.set_device(0)
    import selective_state_space_134_b300 as m3
    m3.lib()
    hbm_peak, _, _ = peaks()
    print(json.dumps({"metric": "decode tokens/s", "unit": "tokens/s", "higher_is_better": True,
                      "workloads": decode_results(m3, hbm_peak)}))


def run_workload(args):
    """One prefill, backward or decode workload alone, optionally resized: a JSON line with its
    tokens/s and roofline (used for profiling runs)."""
    torch.cuda.set_device(0)
    import selective_state_space_134_b300 as m3
    from selective_state_space_134_b300.synth import WORKLOADS
    m3.lib()
    hbm_peak, _, peak_kind = peaks()
    over = {k: v for k, v in (("batch", args.batch), ("nheads", args.heads), ("seqlen", args.seqlen)) if v}
    w = WORKLOADS[args.workload].with_(**over)
    if w.name.startswith("decode"):   # --steps decode calls (one token each), on a state pool with --pooled
        timer = time_decode_pooled if args.pooled else time_decode
        ms_call, k_ms = timer(m3, w, args.steps, args.warmup)
        gbs = decode_bytes(w) / (k_ms * 1e-3) / 1e9
        print(json.dumps({"metric": "decode tokens/s", "workload": w.name, "overrides": over,
                          "pooled": bool(args.pooled), "tokens_per_s": w.batch / (ms_call * 1e-3),
                          "us_per_call": round(ms_call * 1e3, 2), "calls": args.steps,
                          "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                                       "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                                       "algorithmic_bytes": decode_bytes(w), "kernel_ms": k_ms}}))
        return
    if args.backward:
        ms_b, _ = time_backward(m3, w, args.steps, args.warmup)
        print(json.dumps({"metric": "backward tokens/s", "workload": w.name, "overrides": over,
                          "tokens_per_s": w.batch * w.seqlen / (ms_b * 1e-3), "ms_per_step": ms_b}))
        return
    r = time_prefill(m3, w, args.steps, args.warmup, m3.KERNEL_PREFILL_OUTPUT)
    line = prefill_line(m3, w, r, args.steps, hbm_peak, peak_kind)
    line.update({"metric": "prefill tokens/s", "workload": w.name, "overrides": over,
                 "launches_per_step": r["launches"] / args.steps})
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="headline only (no decode / other workloads / oracle)")
    ap.add_argument("--decode-only", action="store_true",
                    help="one JSON line with the four decode workloads only (profiling runs)")
    ap.add_argument("--workload", help="time this prefill or decode workload alone (profiling runs)")
    ap.add_argument("--batch", type=int, default=0, help="with --workload: batch override")
    ap.add_argument("--heads", type=int, default=0, help="with --workload: head-count override")
    ap.add_argument("--seqlen", type=int, default=0, help="with --workload: sequence-length override")
    ap.add_argument("--backward", action="store_true", help="with --workload: time the backward pass")
    ap.add_argument("--pooled", action="store_true", help="with a decode --workload: run it on a state pool")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.workload:
        run_workload(args)
    elif args.decode_only:
        run_decode_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
