"""Host-side pieces of bench.py that decide what a reported number means."""
from __future__ import annotations

import json
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))

import bench  # noqa: E402
from paged_attention_decode_kv_gb300 import workloads as W  # noqa: E402


def test_code_only_ignores_comments_but_not_code():
    a = "int x = 1;  // one\n/* block\n comment */\nint y = 2;\n\n"
    b = "int x = 1;\nint y = 2;"
    assert bench._code_only(a) == b
    assert bench._code_only(a.replace("2", "3")) != b


def test_every_workload_maps_to_an_existing_variant_unit():
    csrc = ROOT / "paged_attention_decode_kv_gb300" / "csrc"
    for name in W.WORKLOADS:
        unit = bench.variant_source(name)
        assert (csrc / unit).exists(), (name, unit)
        assert len(bench.kernel_hash(name)) == 16


def test_recorded_traffic_only_for_matching_code():
    """A stored DRAM figure is reported only while its stamp matches the code
    of that workload's kernel."""
    data = json.loads((ROOT / "profiles" / "traffic.json").read_text())
    for name, entry in data.items():
        got = bench.recorded_traffic(name)
        if entry["kernel_hash"] == bench.kernel_hash(name):
            assert got == entry["dram_bytes_per_launch"]
        else:
            assert got is None
    assert bench.recorded_traffic("no_such_workload") is None


def test_sweep_and_default_workloads_exist():
    assert bench.DEFAULT_WORKLOAD in W.WORKLOADS
    for name in bench.SWEEP:
        assert name in W.WORKLOADS


def test_clock_gate():
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3}
    assert bench.clocks_acceptable(ok)
    assert bench.clocks_acceptable({**ok, "reasons": ["sw_power_cap"], "sm_mhz": 1500.0})
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert not bench.clocks_acceptable({**ok, "reasons": [r]})
    assert not bench.clocks_acceptable({**ok, "sm_mhz": 1200.0})  # locked low, no reason
    assert bench.clocks_acceptable({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0})
