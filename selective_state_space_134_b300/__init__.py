"""B300-native (sm_103a) Mamba-3 layer recurrence: chunked prefill and decode step.

The compute lives in ``libmamba3.so`` (hand-written CUDA behind the C ABI of
``include/mamba3.h``); :mod:`.mamba3` is its ctypes binding and :mod:`.synth`
the seeded synthetic-input generator.
"""
from .mamba3 import (BcNorm, DECODE_GENERIC, DECODE_STREAM, DECODE_TENSOR, KERNEL_BACKWARD, KERNEL_DECODE, KERNEL_PREFILL_OUTPUT, KERNEL_PREFILL_STATE, KERNEL_SEGMENT_PASS, M3_BF16,
                     M3_ERR_INDEX, M3_F16, M3_F32, M3_OK, Mamba3Error, State, decode_last_variant, decode_step,
                     decode_step_pooled, device_status,
                     dims, launch_count, lib,
                     scan_bwd, scan_bwd_workspace, scan_fwd, scan_fwd_workspace, status_string, trace_begin, trace_end)

__all__ = ["BcNorm", "DECODE_GENERIC", "DECODE_STREAM", "DECODE_TENSOR", "KERNEL_BACKWARD", "KERNEL_DECODE", "KERNEL_PREFILL_OUTPUT", "KERNEL_PREFILL_STATE", "KERNEL_SEGMENT_PASS", "M3_BF16",
           "M3_ERR_INDEX", "M3_F16", "M3_F32", "M3_OK", "Mamba3Error", "State", "decode_last_variant", "decode_step", "decode_step_pooled",
           "device_status", "dims", "launch_count",
           "lib", "scan_bwd", "scan_bwd_workspace", "scan_fwd", "scan_fwd_workspace", "status_string", "trace_begin", "trace_end"]
