"""Host-side logic of bench.py on the CPU: algorithmic byte counts and the traffic record lookup."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from selective_state_space_134_b300.build import source_digest  # noqa: E402
from selective_state_space_134_b300.synth import WORKLOADS  # noqa: E402


def test_prefill_bytes_per_token_head():
    # the scope table's formula: e (2PR + 2NR + N/2 + 3), x and y; B, C; theta; dt / A / lambda,
    # every tensor at the input element size e
    w = WORKLOADS["siso_n64"]
    assert bench.bytes_per_token_head(w) == 2 * (2 * 64 + 2 * 64 + 32 + 3) == 582
    w128 = WORKLOADS["siso_n128"]
    assert bench.bytes_per_token_head(w128) == 2 * (2 * 64 + 2 * 128 + 64 + 3) == 902
    w4 = WORKLOADS["mimo_r4"]
    assert bench.bytes_per_token_head(w4) == 2 * (2 * 64 * 4 + 2 * 64 * 4 + 32 + 3) == 2118
    wl = WORKLOADS["long_n128_r4"]
    assert bench.bytes_per_token_head(wl) == 2 * (2 * 64 * 4 + 2 * 128 * 4 + 64 + 3) == 3206
    wt = WORKLOADS["tiny_f32"]
    assert bench.bytes_per_token_head(wt) == 4 * (2 * 16 + 2 * 16 + 8 + 3) == 300
    # grouped B / C: 4 groups of 8 heads read a quarter of the B and C bytes per head
    assert bench.bytes_per_token_head(w, groups=4) == 2 * (2 * 64 + 2 * 64 / 8 + 32 + 3)
    # whole step: every (token, head) (305 MB for siso_n64) plus the final state and carry (2 MB)
    bh = w.batch * w.nheads
    assert bench.prefill_bytes(w) == w.batch * w.seqlen * w.nheads * 582 + bh * 64 * 64 * 4 + bh * (64 + 64) * 2
    assert 307e6 < bench.prefill_bytes(w) < 308e6
    # an fp32 y moves 2 P R more bytes per (token, head) with bf16 inputs, none with fp32 inputs
    assert bench.y_surplus_per_token_head(w) == 2 * 64
    assert bench.y_surplus_per_token_head(w4) == 2 * 64 * 4
    assert bench.y_surplus_per_token_head(w, y_bytes=2) == 0
    assert bench.y_surplus_per_token_head(wt) == 0


def test_decode_bytes_per_call():
    # per head: state read + write 8 N P, carry read + write, token inputs, y at the input size
    w = WORKLOADS["decode_n64_r4"]
    bh = w.batch * w.nheads
    per_head = 8 * 64 * 64 + 2 * 2 * 4 * (64 + 64) + 2 * (4 * 64 + 2 * 4 * 64 + 32 + 3) + 2 * 4 * 64
    assert bench.decode_bytes(w) == bh * per_head
    assert 302e6 < bench.decode_bytes(w) < 304e6    # 303 MB per call
    assert bench.decode_y_surplus(w) == bh * 2 * 4 * 64


def test_prefill_line_reports_the_whole_step():
    # a three-launch step: the whole-step fraction uses the step time, the output pass's own rate
    # is reported beside it
    w = WORKLOADS["long_n128_r4"]
    res = {"ms": 2 * 13.7, "traced": (2, 2 * 10.5)}
    line = bench.prefill_line(None, w, res, 2, 6503.1, "measured")
    algo = bench.prefill_bytes(w)
    rf = line["roofline"]
    assert rf["algorithmic_bytes"] == algo
    assert abs(rf["achieved"] - algo / 13.7e-3 / 1e9) < 0.1
    assert abs(rf["frac"] - algo / 13.7e-3 / 1e9 / 6503.1) < 1e-4
    assert abs(rf["output_pass"]["achieved"] - algo / 10.5e-3 / 1e9) < 0.1
    assert rf["extra_bytes_wide_y"] == w.token_heads * 2 * 64 * 4


def test_traffic_lookup_requires_the_current_source_digest(tmp_path, monkeypatch):
    rec = {"decode/decode_n64_r1": {"source_digest": source_digest("decode"), "dram_bytes_per_launch": 123},
           "decode/decode_n64_r4": {"source_digest": "0" * 16, "dram_bytes_per_launch": 456}}
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("decode", "decode_n64_r1") == 123
    assert bench.traffic_for("decode", "decode_n64_r4") is None       # recorded for other sources
    assert bench.traffic_for("decode", "decode_n128_r1") is None      # never recorded


def test_kernel_digests_cover_their_own_sources():
    # a kernel's traffic record stays valid when only other kernels' sources change
    assert source_digest("prefill_output") != source_digest("decode") != source_digest()
    assert len(source_digest("prefill_output")) == 16
