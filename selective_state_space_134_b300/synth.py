"""Seeded synthetic inputs for the Mamba-3 layer recurrence.

This module only draws random numbers with the distributions of the
workloads and rounds them once to the storage dtype; it holds none of the
recurrence's arithmetic.  Both the CUDA path (through the tests and
``bench.py``) and the CPU oracle read exactly the tensors made here.

Distributions (the same for every workload unless stated):
    x, B, C ~ N(0, 1);  dt = softplus(N(0,1) - shift) with shift 2 (4 for the
    long-context workload, "slow decay");  A = -exp(N(0, 0.5)) read as
    standard deviation 0.5;  lambda = sigmoid(N(0,1));  theta ~ U(-pi, pi);
    h0 = 0 for prefill, h ~ N(0,1) fp32 for decode.
All values are drawn in fp32 with one ``torch.Generator`` seeded per workload
and tensor, then rounded once (round-to-nearest-even) to the workload dtype.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    nheads: int
    seqlen: int
    P: int
    N: int
    R: int
    chunk: int
    dtype: str = "bf16"
    dt_shift: float = 2.0
    seed: int = 0

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def token_heads(self) -> int:
        return self.batch * self.nheads * self.seqlen


# The five workloads of the Mamba-3 recurrence study (shapes of the pages'
# experiments: head dim 64, state 64 vs 128, MIMO rank 4, long sequences).
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 2, 256, 16, 16, 1, 64, "f32", 2.0, 0),
    "siso_n64": Workload("siso_n64", 4, 32, 4096, 64, 64, 1, 64, "bf16", 2.0, 1),
    "siso_n128": Workload("siso_n128", 4, 32, 4096, 64, 128, 1, 64, "bf16", 2.0, 1),
    "mimo_r4": Workload("mimo_r4", 8, 32, 8192, 64, 64, 4, 64, "bf16", 2.0, 2),
    "decode_n64_r1": Workload("decode_n64_r1", 256, 32, 1, 64, 64, 1, 0, "bf16", 2.0, 3),
    "decode_n64_r4": Workload("decode_n64_r4", 256, 32, 1, 64, 64, 4, 0, "bf16", 2.0, 3),
    "decode_n128_r1": Workload("decode_n128_r1", 256, 32, 1, 64, 128, 1, 0, "bf16", 2.0, 3),
    "decode_n128_r4": Workload("decode_n128_r4", 256, 32, 1, 64, 128, 4, 0, "bf16", 2.0, 3),
    "long_n128_r4": Workload("long_n128_r4", 1, 64, 131072, 64, 128, 4, 128, "bf16", 4.0, 4),
}

DECODE_STEPS = 1024      # decode workload: one token per call over this many calls
DECODE_POOL = 64         # distinct per-token input sets, cycled over the calls


def _gen(seed: int, salt: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + salt)
    return g


def _normal(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def token_inputs(w: Workload, device="cpu", lead=None, salt: int = 0) -> dict:
    """Per-token inputs of workload ``w``.

    ``lead`` is the leading shape: (batch, seqlen, nheads) for prefill (the
    default) or (batch, nheads) for a decode token.  Returns x [lead,R,P],
    B, C [lead,R,N], dt, A, lam [lead], theta [lead,N/2] in the workload dtype.
    """
    if lead is None:
        lead = (w.batch, w.seqlen, w.nheads)
    lead = tuple(lead)
    dt_ = DTYPES[w.dtype]
    base = 16 * salt
    out = {}
    out["x"] = _normal(lead + (w.R, w.P), _gen(w.seed, base + 1, device), device).to(dt_)
    out["B"] = _normal(lead + (w.R, w.N), _gen(w.seed, base + 2, device), device).to(dt_)
    out["C"] = _normal(lead + (w.R, w.N), _gen(w.seed, base + 3, device), device).to(dt_)
    z = _normal(lead, _gen(w.seed, base + 4, device), device)
    out["dt"] = torch.nn.functional.softplus(z - w.dt_shift).to(dt_)
    z = _normal(lead, _gen(w.seed, base + 5, device), device)
    out["A"] = (-torch.exp(0.5 * z)).to(dt_)
    z = _normal(lead, _gen(w.seed, base + 6, device), device)
    out["lam"] = torch.sigmoid(z).to(dt_)
    u = torch.rand(lead + (w.N // 2,), generator=_gen(w.seed, base + 7, device), device=device,
                   dtype=torch.float32)
    out["theta"] = ((2.0 * u - 1.0) * math.pi).to(dt_)
    return out


def prefill_inputs(w: Workload, device="cpu") -> dict:
    """Prefill inputs: token tensors [batch, seqlen, nheads, ...]; h0 = 0, no carry."""
    return token_inputs(w, device)


def decode_state(w: Workload, device="cpu") -> dict:
    """Decode state: h ~ N(0,1) fp32 [batch,H,N,P] and a carry (B_prev, x_prev) drawn like B, x."""
    h = _normal((w.batch, w.nheads, w.N, w.P), _gen(w.seed, 900, device), device)
    carry = token_inputs(w, device, lead=(w.batch, w.nheads), salt=63)
    return {"h": h, "B_prev": carry["B"], "x_prev": carry["x"]}


def decode_pool(w: Workload, device="cpu", pool: int = DECODE_POOL) -> list:
    """``pool`` per-token input sets [batch, H, ...], cycled over the decode calls."""
    return [token_inputs(w, device, lead=(w.batch, w.nheads), salt=i + 1) for i in range(pool)]


def to_f64(t: torch.Tensor):
    """Exact widening of stored values to float64 numpy (the oracle's input)."""
    return t.detach().to("cpu", torch.float64).numpy()


def bc_params(w: Workload, device="cpu", seed: int = 0, eps: float = 1e-5) -> dict:
    """Synthetic parameters of the BC normalisation and bias (no trained weights exist here): gains
    U(0.5, 1.5) [H, N] and biases 0.5 N(0, 1) [H, R, N] for B and for C, fp32, and eps."""
    out = {}
    for i, k in enumerate(("B", "C")):
        g = _gen(w.seed + 17 * seed, 500 + 2 * i, device)
        out[f"{k}_weight"] = 0.5 + torch.rand((w.nheads, w.N), generator=g, device=device, dtype=torch.float32)
        g = _gen(w.seed + 17 * seed, 501 + 2 * i, device)
        out[f"{k}_bias"] = 0.5 * _normal((w.nheads, w.R, w.N), g, device)
    out["eps"] = eps
    return out
