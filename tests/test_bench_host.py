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


def test_pair_blocks_cover_every_pair_once_and_reproduce_the_oracle():
    """The CPU baseline splits the pairs over processes; each block through the oracle gives
    exactly its slice of the full problem's outputs (pairs are independent)."""
    import numpy as np
    from matrix_state_nonlinear_gb300.inputs import make_inputs
    from oracle import m2rnn_forward
    for shared in (False, True):
        wl = Workload("blk", 3, 9, 5, 8, 16, h0="uniform", shared_qk=shared)
        arrs = bench.host_arrays(make_inputs(wl, "cpu", 0))
        f = {k: bench._as_f64(v) for k, v in arrs.items()}
        y, HT = m2rnn_forward(f["q"], f["k"], f["v"], f["a"], f["alpha"], f["beta"], f["W"],
                              f["w_r"], f["H0"])
        for parts in (1, 4, 7, 16, 40):
            blocks = bench.pair_blocks(arrs, parts)
            assert len(blocks) <= parts
            seen = np.zeros((3, 5), int)
            for (b0, b1, n0, n1), blk in blocks:
                seen[b0:b1, n0:n1] += 1
                g = {k: bench._as_f64(v) for k, v in blk.items()}
                yb, Hb = m2rnn_forward(g["q"], g["k"], g["v"], g["a"], g["alpha"], g["beta"],
                                       g["W"], g["w_r"], g["H0"])
                assert np.array_equal(yb, y[b0:b1, :, n0:n1])
                assert np.array_equal(Hb, HT[b0:b1, n0:n1])
            assert (seen == 1).all()


def test_oracle_pool_runs_blocks_in_spawned_processes():
    wl = Workload("pool", 2, 6, 3, 8, 16, h0="uniform")
    from matrix_state_nonlinear_gb300.inputs import make_inputs
    pool = bench.OraclePool(2)
    try:
        wall, cpu = pool.run("forward", bench.host_arrays(make_inputs(wl, "cpu", 0)))
    finally:
        pool.close()
    assert wall > 0 and cpu >= 0
    info = bench.host_cores()
    assert info["host_cpu_count"] >= 1 and info["affinity_cores"] >= 1
