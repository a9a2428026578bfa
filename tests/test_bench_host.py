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
    # e (2PR + 2NR + N/2 + 3) + 4PR: x, B, C, theta, dt / A / lambda in bf16, y in fp32
    w = WORKLOADS["siso_n64"]
    assert bench.bytes_per_token_head(w) == 2 * (64 + 2 * 64 + 32 + 3) + 4 * 64
    w4 = WORKLOADS["mimo_r4"]
    assert bench.bytes_per_token_head(w4) == 2 * (64 * 4 + 2 * 64 * 4 + 32 + 3) + 4 * 64 * 4
    # grouped B / C: 4 groups of 8 heads read a quarter of the B and C bytes per head
    assert bench.bytes_per_token_head(w, groups=4) == 2 * (64 + 2 * 64 / 8 + 32 + 3) + 4 * 64
    # whole step: every (token, head) plus the final state and carry
    bh = w.batch * w.nheads
    assert bench.prefill_bytes(w) == w.batch * w.seqlen * w.nheads * bench.bytes_per_token_head(w) + \
        bh * 64 * 64 * 4 + bh * (64 + 64) * 2


def test_decode_bytes_per_call():
    # per head: state read + write 8 N P, carry read + write, token inputs, y (fp32)
    w = WORKLOADS["decode_n64_r4"]
    bh = w.batch * w.nheads
    per_head = 8 * 64 * 64 + 2 * 2 * 4 * (64 + 64) + 2 * (4 * 64 + 2 * 4 * 64 + 32 + 3) + 4 * 4 * 64
    assert bench.decode_bytes(w) == bh * per_head


def test_traffic_lookup_requires_the_current_source_digest(tmp_path, monkeypatch):
    rec = {"decode/decode_n64_r1": {"source_digest": source_digest(), "dram_bytes_per_launch": 123},
           "decode/decode_n64_r4": {"source_digest": "0" * 16, "dram_bytes_per_launch": 456}}
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("decode", "decode_n64_r1") == 123
    assert bench.traffic_for("decode", "decode_n64_r4") is None       # recorded for other sources
    assert bench.traffic_for("decode", "decode_n128_r1") is None      # never recorded
