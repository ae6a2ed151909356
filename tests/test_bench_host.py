"""Host logic of the bench that its reported figures depend on: the algorithmic
bytes per decode launch (the roofline numerator) and the rule that a recorded
ncu traffic figure is reported only for the sources it was taken with."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_decode_launch_bytes_headline():
    # batch 1, Llama3.2-3B layer: |S| records of gate row + up row + down
    # column (3 x 2d bytes), a 4-byte position each, x (2d) in and y (4d) out
    w = synth.WORKLOADS["llama3.2-3b"]
    n = 4096
    assert bench.decode_launch_bytes(w, n, n) == n * 6 * 3072 + 4 * n + 2 * 3072 + 4 * 3072 == 75532288


def test_decode_launch_bytes_batch_counts_the_union_once():
    # B sequences read the union of their sets once, with a position and a
    # sequence mask per record, and B inputs and outputs
    w = synth.WORKLOADS["qwen2.5-3b"]
    u = 6067
    assert bench.decode_launch_bytes(w, u, 4404) == u * 6 * w.d + 8 * u + w.B * 6 * w.d


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    rec = {"k@w": {"dram_bytes_per_launch": 123, "source_hash": bench.kernel_source_hash(), "capture": "cmd"}}
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: rec["k@w"]["source_hash"])
    assert bench.recorded_traffic("k@w") == (123, "cmd")
    assert bench.recorded_traffic("other@w") == (None, "no capture recorded for this kernel")
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.recorded_traffic("k@w") == (None, "kernel changed since the capture")

