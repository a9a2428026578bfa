"""Python binding of libmamba3.so (the C ABI in include/mamba3.h).

Argument marshalling only: tensors are passed as raw device pointers and every
step of the recurrence runs in the library's CUDA kernels.  PyTorch provides
device memory and the current stream.  There is no fallback: if the library is
missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmamba3.so")

M3_OK, M3_ERR_INVALID_ARG, M3_ERR_UNSUPPORTED, M3_ERR_WORKSPACE, M3_ERR_CUDA, M3_ERR_TIMEOUT, M3_ERR_INDEX = range(7)
M3_F32, M3_BF16, M3_F16 = 0, 1, 2
_DTYPE_CODE = {torch.float32: M3_F32, torch.bfloat16: M3_BF16, torch.float16: M3_F16}


class m3_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("seqlen", ctypes.c_int), ("nheads", ctypes.c_int),
                ("headdim", ctypes.c_int), ("dstate", ctypes.c_int), ("rank", ctypes.c_int),
                ("chunk", ctypes.c_int), ("dtype", ctypes.c_int), ("ngroups", ctypes.c_int),
                ("ydtype", ctypes.c_int)]


class m3_state(ctypes.Structure):
    _fields_ = [("h", ctypes.c_void_p), ("B_prev", ctypes.c_void_p), ("x_prev", ctypes.c_void_p)]


class m3_bc_norm(ctypes.Structure):
    _fields_ = [("B_weight", ctypes.c_void_p), ("B_bias", ctypes.c_void_p), ("C_weight", ctypes.c_void_p),
                ("C_bias", ctypes.c_void_p), ("eps", ctypes.c_float)]


@dataclass
class BcNorm:
    """BC normalisation and bias: every (token, head, rank) row v of B (C) becomes
    v / sqrt(mean(v^2) + eps) * weight[h] + bias[h, r].  weight [H, N], bias [H, R, N] fp32 device
    tensors, or None (gain 1 / no bias)."""
    B_weight: Optional[torch.Tensor] = None
    B_bias: Optional[torch.Tensor] = None
    C_weight: Optional[torch.Tensor] = None
    C_bias: Optional[torch.Tensor] = None
    eps: float = 1e-6

    def c(self) -> m3_bc_norm:
        for t in (self.B_weight, self.B_bias, self.C_weight, self.C_bias):
            if t is not None and t.dtype != torch.float32:
                raise ValueError("BC gains and biases are fp32")
        return m3_bc_norm(_ptr(self.B_weight), _ptr(self.B_bias), _ptr(self.C_weight), _ptr(self.C_bias),
                          float(self.eps))


class m3_token_inputs(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in ("x", "B", "C", "dt", "A", "lam", "theta")]


class m3_grads_in(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in ("dy", "dh_out", "dB_prev_out", "dx_prev_out")]


class m3_grads_out(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in ("dx", "dB", "dC", "ddt", "dA", "dlambda", "dtheta", "dh0", "dB_prev",
                                              "dx_prev")]


class Mamba3Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None


def lib() -> ctypes.CDLL:
    """Loads libmamba3.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m selective_state_space_134_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, dp, sp = ctypes.c_void_p, ctypes.POINTER(m3_dims), ctypes.POINTER(m3_state)
        L.mamba3_scan_fwd_workspace.argtypes = [dp, ctypes.POINTER(ctypes.c_size_t)]
        L.mamba3_scan_fwd_workspace.restype = ctypes.c_int
        L.mamba3_scan_fwd.argtypes = [dp] + [vp] * 7 + [sp, vp, sp, vp, ctypes.c_size_t, vp]
        L.mamba3_scan_fwd.restype = ctypes.c_int
        L.mamba3_decode_step.argtypes = [dp] + [vp] * 7 + [sp, vp, vp]
        L.mamba3_decode_step.restype = ctypes.c_int
        L.mamba3_decode_step_pooled.argtypes = [dp] + [vp] * 8 + [sp, ctypes.c_int, vp, vp]
        L.mamba3_decode_step_pooled.restype = ctypes.c_int
        L.mamba3_device_status.argtypes = [vp]
        L.mamba3_device_status.restype = ctypes.c_int
        L.mamba3_status_string.argtypes = [ctypes.c_int]
        L.mamba3_status_string.restype = ctypes.c_char_p
        L.mamba3_launch_count.argtypes = []
        L.mamba3_launch_count.restype = ctypes.c_uint64
        L.mamba3_trace_begin.argtypes = [ctypes.c_int, ctypes.c_int]
        L.mamba3_trace_begin.restype = ctypes.c_int
        L.mamba3_trace_end.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_double)]
        L.mamba3_trace_end.restype = ctypes.c_int
        L.mamba3_scan_fwd_staged_workspace.argtypes = [dp, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]
        L.mamba3_scan_fwd_staged_workspace.restype = ctypes.c_int
        ip = ctypes.POINTER(m3_token_inputs)
        L.mamba3_scan_fwd_staged.argtypes = [dp, ip, ip, vp, vp, sp, sp, vp, vp, ctypes.c_size_t, ctypes.c_int,
                                             vp, vp]
        L.mamba3_scan_fwd_staged.restype = ctypes.c_int
        bp = ctypes.POINTER(m3_bc_norm)
        L.mamba3_scan_fwd_bc.argtypes = [dp] + [vp] * 7 + [bp, sp, vp, sp, vp, ctypes.c_size_t, vp]
        L.mamba3_scan_fwd_bc.restype = ctypes.c_int
        L.mamba3_decode_step_bc.argtypes = [dp] + [vp] * 7 + [bp, sp, vp, vp]
        L.mamba3_decode_step_bc.restype = ctypes.c_int
        L.mamba3_scan_bwd_workspace.argtypes = [dp, ctypes.POINTER(ctypes.c_size_t)]
        L.mamba3_scan_bwd_workspace.restype = ctypes.c_int
        L.mamba3_scan_bwd.argtypes = [dp, ctypes.POINTER(m3_token_inputs), sp, ctypes.POINTER(m3_grads_in),
                                      ctypes.POINTER(m3_grads_out), vp, ctypes.c_size_t, vp]
        L.mamba3_scan_bwd.restype = ctypes.c_int
        L.mamba3_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        L.mamba3_selftest_wait_timeout.restype = ctypes.c_int
        L.mamba3_decode_last_variant.argtypes = []
        L.mamba3_decode_last_variant.restype = ctypes.c_int
        L.mamba3_version.argtypes = []
        L.mamba3_version.restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().mamba3_status_string(int(status)).decode()


def launch_count() -> int:
    return int(lib().mamba3_launch_count())


def _check(status: int, what: str):
    if status != M3_OK:
        raise Mamba3Error(status, what)


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


@dataclass
class State:
    """Recurrent state: h [b,H,N,P] fp32; carry B_prev [b,H,R,N], x_prev [b,H,R,P] (input dtype)."""
    h: torch.Tensor
    B_prev: Optional[torch.Tensor] = None
    x_prev: Optional[torch.Tensor] = None

    def c(self) -> m3_state:
        return m3_state(_ptr(self.h), _ptr(self.B_prev), _ptr(self.x_prev))

    @staticmethod
    def zeros(batch, nheads, P, N, R, dtype, device="cuda") -> "State":
        return State(torch.zeros(batch, nheads, N, P, dtype=torch.float32, device=device),
                     torch.zeros(batch, nheads, R, N, dtype=dtype, device=device),
                     torch.zeros(batch, nheads, R, P, dtype=dtype, device=device))


def _code(dtype) -> int:
    return _DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)


def dims(batch, seqlen, nheads, P, N, R, dtype, chunk=0, ngroups=0, ydtype=torch.float32) -> m3_dims:
    """ngroups: B / C groups of heads (0 = one B and C per head); ydtype: element type of y."""
    return m3_dims(batch, seqlen, nheads, P, N, R, chunk, _code(dtype), ngroups, _code(ydtype))


def _groups(H: int, G: int) -> int:
    # the head axis of B / C: H = one per head (ngroups 0), else G groups
    return 0 if G == H else G


def scan_fwd_workspace(d: m3_dims) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().mamba3_scan_fwd_workspace(ctypes.byref(d), ctypes.byref(n)), "mamba3_scan_fwd_workspace")
    return int(n.value)


def scan_fwd(x, B, C, dt, A, lam, theta, state_in: Optional[State] = None,
             state_out: Optional[State] = None, chunk: int = 0, y: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None, stream=None, y_dtype=torch.float32,
             bc: Optional[BcNorm] = None) -> torch.Tensor:
    """Chunked prefill.  x [b,L,H,R,P]; B, C [b,L,H,R,N] (or [b,L,G,R,N]: G groups of heads);
    dt, A, lam [b,L,H]; theta [b,L,H,N/2].

    Returns y [b,L,H,R,P] of ``y_dtype`` (fp32, fp16 or bf16; the dtype of ``y`` when given).
    ``state_out`` (may be ``state_in``) receives the final state and carry.  The workspace is
    allocated here through torch unless given.  ``bc``: BC normalisation and bias in front of the
    recurrence (mamba3_scan_fwd_bc).
    """
    b, L, H, R, P = x.shape
    N = B.shape[-1]
    if y is not None:
        y_dtype = y.dtype
    d = dims(b, L, H, P, N, R, x.dtype, chunk, _groups(H, B.shape[2]), y_dtype)
    if y is None:
        y = torch.empty(x.shape, dtype=y_dtype, device=x.device)
    ws_bytes = scan_fwd_workspace(d)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    st_in = state_in.c() if state_in is not None else None
    st_out = state_out.c() if state_out is not None else None
    tail = (ctypes.byref(st_in) if st_in is not None else None, _ptr(y),
            ctypes.byref(st_out) if st_out is not None else None,
            _ptr(workspace), workspace.numel() if workspace is not None else 0, _stream_ptr(stream))
    head = (ctypes.byref(d), _ptr(x), _ptr(B), _ptr(C), _ptr(dt), _ptr(A), _ptr(lam), _ptr(theta))
    if bc is None:
        _check(lib().mamba3_scan_fwd(*head, *tail), "mamba3_scan_fwd")
    else:
        bcs = bc.c()
        _check(lib().mamba3_scan_fwd_bc(*head, ctypes.byref(bcs), *tail), "mamba3_scan_fwd_bc")
    return y


def decode_step(x, B, C, dt, A, lam, theta, state: State, y: Optional[torch.Tensor] = None,
                stream=None, y_dtype=torch.float32, bc: Optional[BcNorm] = None) -> torch.Tensor:
    """One token for every (b, h).  x [b,H,R,P]; B, C [b,H,R,N] (or [b,G,R,N]: G groups of heads);
    dt, A, lam [b,H]; theta [b,H,N/2].

    Updates ``state`` in place and returns y [b,H,R,P] of ``y_dtype`` (the dtype of ``y`` when given).
    """
    b, H, R, P = x.shape
    N = B.shape[-1]
    if y is not None:
        y_dtype = y.dtype
    d = dims(b, 1, H, P, N, R, x.dtype, 0, _groups(H, B.shape[1]), y_dtype)
    if y is None:
        y = torch.empty(x.shape, dtype=y_dtype, device=x.device)
    st = state.c()
    head = (ctypes.byref(d), _ptr(x), _ptr(B), _ptr(C), _ptr(dt), _ptr(A), _ptr(lam), _ptr(theta))
    if bc is None:
        _check(lib().mamba3_decode_step(*head, ctypes.byref(st), _ptr(y), _stream_ptr(stream)), "mamba3_decode_step")
    else:
        bcs = bc.c()
        _check(lib().mamba3_decode_step_bc(*head, ctypes.byref(bcs), ctypes.byref(st), _ptr(y), _stream_ptr(stream)),
               "mamba3_decode_step_bc")
    return y


def decode_step_pooled(x, B, C, dt, A, lam, theta, slot: torch.Tensor, pool: State,
                       y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """mamba3_decode_step_pooled: one token per batch row, states in a pool.

    slot [b] int32 on the device: pool slot of each row (< 0: inactive row, left untouched).
    pool: State with h [S,H,N,P], B_prev [S,H,R,N], x_prev [S,H,R,P], updated in place.
    Returns y [b,H,R,P] (fp32; rows of inactive slots keep what ``y`` held).
    """
    b, H, R, P = x.shape
    N = B.shape[-1]
    if slot.dtype != torch.int32:
        raise ValueError("slot must be int32")
    d = dims(b, 1, H, P, N, R, x.dtype, 0, _groups(H, B.shape[1]), y.dtype if y is not None else torch.float32)
    if y is None:
        y = torch.zeros(x.shape, dtype=torch.float32, device=x.device)
    rc = lib().mamba3_decode_step_pooled(ctypes.byref(d), _ptr(slot), _ptr(x), _ptr(B), _ptr(C), _ptr(dt),
                                         _ptr(A), _ptr(lam), _ptr(theta), ctypes.byref(pool.c()),
                                         int(pool.h.shape[0]), _ptr(y), _stream_ptr(stream))
    _check(rc, "mamba3_decode_step_pooled")
    return y


KERNEL_PREFILL_STATE, KERNEL_SEGMENT_PASS, KERNEL_PREFILL_OUTPUT, KERNEL_DECODE, KERNEL_BACKWARD = range(5)


def scan_bwd_workspace(d: m3_dims) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().mamba3_scan_bwd_workspace(ctypes.byref(d), ctypes.byref(n)), "mamba3_scan_bwd_workspace")
    return int(n.value)


def scan_bwd(x, B, C, dt, A, lam, theta, dy, state_in: Optional[State] = None, dh_out=None, dB_prev_out=None,
             dx_prev_out=None, workspace: Optional[torch.Tensor] = None, grads: Optional[dict] = None,
             stream=None) -> dict:
    """mamba3_scan_bwd: gradients of sum(dy * y) (+ the final state's and carry's terms) with respect
    to the prefill's inputs.  Returns a dict of fp32 tensors: x, B, C, dt, A, lam, theta, h0, Bprev,
    xprev (allocated through torch unless ``grads`` holds them)."""
    b, L, H, R, P = x.shape
    N = B.shape[-1]
    d = dims(b, L, H, P, N, R, x.dtype, 0, _groups(H, B.shape[2]))
    need = scan_bwd_workspace(d)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    if grads is None:
        f = lambda t: torch.empty(t.shape, dtype=torch.float32, device=x.device)
        grads = {"x": f(x), "B": f(B), "C": f(C), "dt": f(dt), "A": f(A), "lam": f(lam), "theta": f(theta),
                 "h0": torch.empty((b, H, N, P), dtype=torch.float32, device=x.device),
                 "Bprev": torch.empty((b, H, R, N), dtype=torch.float32, device=x.device),
                 "xprev": torch.empty((b, H, R, P), dtype=torch.float32, device=x.device)}
    ins = m3_token_inputs(*(_ptr(t) for t in (x, B, C, dt, A, lam, theta)))
    gin = m3_grads_in(_ptr(dy), _ptr(dh_out), _ptr(dB_prev_out), _ptr(dx_prev_out))
    gout = m3_grads_out(*(_ptr(grads.get(k)) for k in ("x", "B", "C", "dt", "A", "lam", "theta", "h0", "Bprev",
                                                        "xprev")))
    st = state_in.c() if state_in is not None else None
    rc = lib().mamba3_scan_bwd(ctypes.byref(d), ctypes.byref(ins), ctypes.byref(st) if st is not None else None,
                               ctypes.byref(gin), ctypes.byref(gout), _ptr(workspace),
                               workspace.numel() if workspace is not None else 0, _stream_ptr(stream))
    _check(rc, "mamba3_scan_bwd")
    return grads


def trace_begin(kernel: int, max_launches: int):
    """Brackets the next ``max_launches`` launches of ``kernel`` with CUDA events (library-side)."""
    _check(lib().mamba3_trace_begin(int(kernel), int(max_launches)), "mamba3_trace_begin")


def trace_end():
    """Returns (launches, total_ms) of the traced kernel and stops tracing."""
    n, ms = ctypes.c_int(0), ctypes.c_double(0.0)
    _check(lib().mamba3_trace_end(ctypes.byref(n), ctypes.byref(ms)), "mamba3_trace_end")
    return int(n.value), float(ms.value)


DECODE_GENERIC, DECODE_STREAM, DECODE_TENSOR = range(3)


def decode_last_variant() -> int:
    """Which decode kernel (DECODE_GENERIC / DECODE_STREAM / DECODE_TENSOR) served the last decode call."""
    return int(lib().mamba3_decode_last_variant())


def device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status (M3_OK, M3_ERR_TIMEOUT or
    M3_ERR_INDEX)."""
    return int(lib().mamba3_device_status(_stream_ptr(stream)))


def scan_fwd_noalloc(x, B, C, dt, A, lam, theta, state_in: Optional[State] = None,
                     state_out: Optional[State] = None, chunk: int = 0, y: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    """mamba3_scan_fwd_noalloc: the prefill with the library's static scratch instead of a workspace.

    For callers that cannot allocate device memory (see include/mamba3.h); y is still passed in
    or, as a convenience of this binding, allocated here through torch.
    """
    L_ = lib()
    fn = L_.mamba3_scan_fwd_noalloc
    fn.argtypes = [ctypes.POINTER(m3_dims)] + [ctypes.c_void_p] * 7 + \
        [ctypes.POINTER(m3_state), ctypes.c_void_p, ctypes.POINTER(m3_state), ctypes.c_void_p]
    fn.restype = ctypes.c_int
    b, L, H, R, P = x.shape
    N = B.shape[-1]
    d = dims(b, L, H, P, N, R, x.dtype, chunk, _groups(H, B.shape[2]), y.dtype if y is not None else torch.float32)
    if y is None:
        y = torch.empty(x.shape, dtype=torch.float32, device=x.device)
    st_in = state_in.c() if state_in is not None else None
    st_out = state_out.c() if state_out is not None else None
    rc = fn(ctypes.byref(d), _ptr(x), _ptr(B), _ptr(C), _ptr(dt), _ptr(A), _ptr(lam), _ptr(theta),
            ctypes.byref(st_in) if st_in is not None else None, _ptr(y),
            ctypes.byref(st_out) if st_out is not None else None, _stream_ptr(stream))
    _check(rc, "mamba3_scan_fwd_noalloc")
    return y


TOKEN_KEYS = ("x", "B", "C", "dt", "A", "lam", "theta")
_side_streams = {}


def _side_stream(device) -> "torch.cuda.Stream":
    """A second stream per device for the copies out of scan_fwd_staged."""
    key = torch.device(device).index if torch.device(device).index is not None else torch.cuda.current_device()
    if key not in _side_streams:
        _side_streams[key] = torch.cuda.Stream(device=key)
    return _side_streams[key]


def scan_fwd_staged_workspace(d: m3_dims, slices: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().mamba3_scan_fwd_staged_workspace(ctypes.byref(d), int(slices), ctypes.byref(n)),
           "mamba3_scan_fwd_staged_workspace")
    return int(n.value)


def scan_fwd_staged(host: dict, dev: dict, host_y: torch.Tensor, dev_y: torch.Tensor,
                    state_out: Optional[State] = None, host_h: Optional[torch.Tensor] = None,
                    state_in: Optional[State] = None, slices: int = 4, workspace: Optional[torch.Tensor] = None,
                    stream=None, copy_stream=None):
    """mamba3_scan_fwd_staged: the prefill from pinned host tensors to host tensors, the copies
    overlapped with the kernels over `slices` batch slices.

    ``host`` / ``dev``: dicts of the seven token inputs (keys x, B, C, dt, A, lam, theta) in pinned host
    memory and same-shaped device staging buffers.  ``host_y`` / ``dev_y``: y in host and device memory.
    ``state_out`` (device) receives the final state and carry, copied to ``host_h`` when given.
    Returns after enqueueing; synchronise ``copy_stream`` before reading the host outputs.
    """
    x = host["x"]
    b, L, H, R, P = x.shape
    N = host["B"].shape[-1]
    d = dims(b, L, H, P, N, R, x.dtype, 0, _groups(H, host["B"].shape[2]), dev_y.dtype)
    need = scan_fwd_staged_workspace(d, slices)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev_y.device)
    hi = m3_token_inputs(*(_ptr(host[k]) for k in TOKEN_KEYS))
    di = m3_token_inputs(*(_ptr(dev[k]) for k in TOKEN_KEYS))
    st_in = state_in.c() if state_in is not None else None
    st_out = state_out.c() if state_out is not None else None
    if copy_stream is None:
        copy_stream = _side_stream(dev_y.device)
    rc = lib().mamba3_scan_fwd_staged(ctypes.byref(d), ctypes.byref(hi), ctypes.byref(di), _ptr(host_y), _ptr(dev_y),
                                      ctypes.byref(st_in) if st_in is not None else None,
                                      ctypes.byref(st_out) if st_out is not None else None, _ptr(host_h),
                                      _ptr(workspace), workspace.numel() if workspace is not None else 0,
                                      int(slices), _stream_ptr(stream), _stream_ptr(copy_stream))
    _check(rc, "mamba3_scan_fwd_staged")
