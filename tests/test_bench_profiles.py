"""The recorded DRAM traffic bench.py reports as roofline.traffic.

profiles/traffic.json holds, per operand kind and workload, the gate/up
kernel's DRAM bytes per launch from an ncu capture and the key of the
kernel sources it was taken on. bench.py must use a figure only while the
current sources still have that key, and report null otherwise.
"""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_traffic_entries_are_well_formed():
    entries = bench.traffic_entries()
    assert entries, bench.TRAFFIC_FILE
    for (quant, workload), e in entries.items():
        assert quant in (None, "fp8", "nvfp4")
        assert workload in bench.WORKLOADS
        assert int(e["dram_bytes_per_launch"]) > 0
        key = e["kernel_source_sha256"]
        assert len(key) == 16 and int(key, 16) >= 0
        assert os.path.exists(os.path.join(ROOT, "profiles", e["summary"])), e["summary"]


@pytest.mark.parametrize("quant,workload", sorted(bench.traffic_entries(),
                                                  key=lambda q: (str(q[0]), q[1])))
def test_traffic_is_used_only_for_the_sources_it_was_taken_on(quant, workload):
    e = bench.traffic_entries()[(quant, workload)]
    got = bench.recorded_traffic(quant, workload)
    if e["kernel_source_sha256"] == bench.kernel_source_key():
        assert got == float(e["dram_bytes_per_launch"])
    else:
        assert got is None


def test_stale_key_gives_null(tmp_path, monkeypatch):
    d = {"entries": [{"quant": "bf16", "workload": "mixtral_8x7b_prefill", "kernel": "gate_up",
                      "dram_bytes_per_launch": 123, "kernel_source_sha256": "0" * 16,
                      "summary": "x.md"}]}
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(d))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(p))
    assert bench.recorded_traffic(None, "mixtral_8x7b_prefill") is None
    d["entries"][0]["kernel_source_sha256"] = bench.kernel_source_key()
    p.write_text(json.dumps(d))
    assert bench.recorded_traffic(None, "mixtral_8x7b_prefill") == 123.0
    assert bench.recorded_traffic("fp8", "mixtral_8x7b_prefill") is None


def test_source_key_format():
    """The key is the first 16 hex digits of a sha256."""
    key = bench.kernel_source_key()
    assert key is not None and len(key) == 16
    int(key, 16)
