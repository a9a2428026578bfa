"""Benchmark of the Mamba-3 layer recurrence on B300: prefill and decode tokens/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--quick] [--decode-only]

A step is one mamba3_scan_fwd over the SISO bf16 prefill workload (batch 4,
32 heads, L = 4096, P = 64, N = 64, R = 1): the prefill hot path end to end
(prefix + RoPE, in-chunk contraction, state passing, outputs and final
state).  `value` = prefill tokens/s (batch x L / time; a token covers every
head), inputs resident in HBM and larger than L2 (no flush needed).  The same
line carries the decode-step measurement (batch 256, 32 heads, one token per
call over 1024 calls; also N = 64, R = 4 on a 512-slot state pool), the other
prefill workloads (N = 128, MIMO R = 4, long context, and the headline shape
with grouped B / C), the roofline of the dominant kernel (timed live through
the library's event tracing; `traffic` from profiles/traffic.json while the
library sources match its digest), the end-to-end figure through host
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
    if trace_kernel is not None:
        m3.trace_begin(trace_kernel, steps)
    n0 = m3.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    launches = m3.launch_count() - n0
    ms = e0.elapsed_time(e1)
    traced = m3.trace_end() if trace_kernel is not None else (0, 0.0)
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
                     "traffic": traffic_for("prefill_output", w.name + (f"_g{groups}" if groups else "")),
                     "algorithmic_bytes": algo,
                     "extra_bytes_wide_y": int(w.token_heads * y_surplus_per_token_head(w, y_bytes)),
                     "y_bytes": y_bytes,
                     "output_pass": {"kernel_ms": k_ms, "achieved": round(achieved_k, 1),
                                     "frac": round(achieved_k / hbm_peak, 4)},
                     "peak_source": peak_kind},
    }


def traffic_for(kernel, workload):
    """ncu DRAM bytes per launch recorded under profiles/ for the current kernel source, else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        from selective_state_space_134_b300.build import source_digest
        r = rec.get(f"{kernel}/{workload}")
        if r and r.get("source_digest") == source_digest():
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
    m3.trace_begin(m3.KERNEL_DECODE, calls)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(calls):
        m3.decode_step(*argsets[i % len(pool)], state=state, y=ys[i % len(pool)])
    e1.record()
    torch.cuda.synchronize()
    n_tr, tr_ms = m3.trace_end()
    assert m3.device_status() == m3.M3_OK
    return e0.elapsed_time(e1) / calls, tr_ms / max(n_tr, 1)


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
    m3.trace_begin(m3.KERNEL_DECODE, calls)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(calls):
        m3.decode_step_pooled(*argsets[i % len(toks)], slot=slot, pool=pool, y=ys[i % len(toks)])
    e1.record()
    torch.cuda.synchronize()
    n_tr, tr_ms = m3.trace_end()
    assert m3.device_status() == m3.M3_OK
    return e0.elapsed_time(e1) / calls, tr_ms / max(n_tr, 1)


def e2e_prefill(m3, w, inp, steps, warmup, slices=16):
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


def cpu_oracle_rate(w, inp, max_seconds=12.0):
    """The fp64 CPU oracle on a bounded sample of the workload, all host cores; tokens/s.

    The sample is 2 x cores whole (b, h) sequences, scanned again and again until
    about `max_seconds` of wall time have passed."""
    import oracle
    from selective_state_space_134_b300.synth import to_f64
    cores = os.cpu_count() or 1
    nseq = max(1, min(w.batch * w.nheads, 2 * cores))
    pairs = [(i // w.nheads, i % w.nheads) for i in range(nseq)]
    stack = {k: torch.cat([inp[k][b:b + 1, :, h:h + 1] for b, h in pairs], 0) for k in KEYS}
    arrs = [to_f64(stack[k]) for k in KEYS]
    threads = min(cores, nseq)
    reps = 0
    t = time.perf_counter()
    while True:
        oracle.scan(*arrs, nthreads=threads)
        reps += 1
        sec = time.perf_counter() - t
        if sec >= max_seconds:
            break
    tok_heads = reps * nseq * w.seqlen
    return {"value": tok_heads / w.nheads / sec, "unit": "tokens/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{nseq} of {w.batch * w.nheads} (b,h) sequences x {w.seqlen} tokens of {w.name}, "
                      f"scanned {reps} times ({sec:.1f} s); tokens/s counts a token as all {w.nheads} heads",
            "seconds": round(sec, 2)}


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
    m3.trace_begin(m3.KERNEL_PREFILL_OUTPUT, args.steps)
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
    traced = m3.trace_end()
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
        for name, steps in (("siso_n128", 20), ("mimo_r4", 5), ("long_n128_r4", 2)):
            wp = WORKLOADS[name]
            r = time_prefill(m3, wp, steps, 1, m3.KERNEL_PREFILL_OUTPUT)
            pre[name] = prefill_line(m3, wp, r, steps, hbm_peak, peak_kind)
            pre[name]["launches_per_step"] = r["launches"] / steps
            del r
            torch.cuda.empty_cache()
        # grouped B / C: siso_n64 with one B and C per 8 heads
        wp = WORKLOADS[HEADLINE]
        r = time_prefill(m3, wp, 20, 1, m3.KERNEL_PREFILL_OUTPUT, groups=4)
        pre["siso_n64_grouped_g4"] = prefill_line(m3, wp, r, 20, hbm_peak, peak_kind, groups=4)
        pre["siso_n64_grouped_g4"]["launches_per_step"] = r["launches"] / 20
        del r
        torch.cuda.empty_cache()
        extra["prefill"] = pre

    e2e = e2e_prefill(m3, w, inp, max(2, min(args.steps, 10)), 1) if rank == 0 else None
    cpu = cpu_oracle_rate(w, inp) if (rank == 0 and ws == 1 and not args.quick) else None

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
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from selective_state_space_134_b300.synth import WORKLOADS, prefill_inputs, to_f64
    w = WORKLOADS[HEADLINE]
    cores = os.cpu_count() or 1
    nseq = min(cores, w.batch * w.nheads)
    inp = prefill_inputs(w.with_(batch=1, nheads=nseq), "cpu")
    arrs = [to_f64(inp[k]) for k in KEYS]
    for _ in range(args.warmup):
        oracle.scan(*(a[:, :256] for a in arrs), nthreads=nseq)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.scan(*arrs, nthreads=nseq)
    sec = (time.perf_counter() - t) / args.steps
    value = nseq * w.seqlen / w.nheads / sec
    sample = (f"per step {nseq} (b,h) sequences x {w.seqlen} tokens of {HEADLINE} (of {w.batch * w.nheads}); "
              f"tokens/s counts a token as all {w.nheads} heads")
    print(json.dumps({
        "impl": "reference", "metric": "prefill tokens/s", "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{HEADLINE}: SISO bf16 prefill, batch {w.batch}, heads {w.nheads}, "
                               f"L={w.seqlen}, P={w.P}, N={w.N}, R={w.R}"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nseq, "kind": "oracle", "sample": sample},
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="headline only (no decode / other workloads / oracle)")
    ap.add_argument("--decode-only", action="store_true",
                    help="one JSON line with the four decode workloads only (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.decode_only:
        run_decode_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
