"""Host-side logic of bench.py (no GPU): the DRAM-traffic record is scaled by the units a
launch processes, and it is withheld once the kernel's source differs from the captured one."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from matrix_state_nonlinear_gb300.inputs import WORKLOADS, Workload  # noqa: E402


def _records():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        return json.load(fh)


def test_every_record_names_its_sources_and_units():
    for name, rec in _records().items():
        assert name in bench.KERNEL_SOURCES, name
        assert rec["units"] > 0 and rec["bytes_per_launch"] > 0, name
        assert len(rec["source_sha256"]) == 64, name


def test_traffic_scales_with_units_and_needs_the_captured_source(monkeypatch):
    rec = _records()["mma_sync_pipelined"]
    wl = WORKLOADS["b8_t16384_n16_k64_v64"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda name: rec["source_sha256"])
    assert bench.measured_traffic("mma_sync_pipelined", wl) == rec["bytes_per_launch"] * wl.units / rec["units"]
    half = Workload("half", wl.B // 2, wl.T, wl.N, wl.K, wl.V)
    assert bench.measured_traffic("mma_sync_pipelined", half) == rec["bytes_per_launch"] * half.units / rec["units"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda name: "0" * 64)
    assert bench.measured_traffic("mma_sync_pipelined", wl) is None
    assert bench.measured_traffic("no_such_kernel", wl) is None
