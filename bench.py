"""Throughput of the M²RNN forward recurrence on GB300: tokens·heads per second.

One step = one full forward pass (gate, rank-1 write, H W contraction, tanh,
gate lerp, readout, writeback) over the whole workload, inputs resident in HBM.
Default workload: the 16K-context training shape B=8, T=16384, N=16, K=V=64,
bf16 operands / fp32 state.  Inputs (0.81 GB of q, k, v, a) are larger than the
129 MB L2, so no flush is needed between timed steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Under torchrun (N > 1) every rank runs its own replica of the workload (the
(batch, head) pairs are independent; there is no exchange step), and the value
is the units of all ranks divided by the slowest rank's time.
`--impl reference` times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "M²RNN fwd tokens·heads/s at K=V=64,T=16K; % of MMA/HBM roofline"
UNIT = "tokens·heads/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=None)
    ap.add_argument("--variant", type=int, default=0)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override B of the workload (smaller cases for profiling)")
    ap.add_argument("--seq", type=int, default=None,
                    help="override T of the workload (smaller cases for profiling)")
    ap.add_argument("--heads", type=int, default=None,
                    help="override N of the workload (fewer pairs)")
    ap.add_argument("--pass", dest="which", default="forward",
                    choices=["forward", "train", "decode", "block"],
                    help="forward: the forward pass (default); train: the state-keeping "
                         "forward plus the backward pass; decode: one-token decode steps; "
                         "block: conv/SiLU prologue + forward + gate/RMSNorm epilogue")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


KERNEL_SOURCES = {
    "mma_sync_rowwarp": ["m2rnn_bf16_mma.cu"],
    "mma_sync_pipelined": ["m2rnn_bf16_pipe.cu"],
    "tcgen05_k128_v128": ["m2rnn_bf16_tc5.cu"],
    "tcgen05_k128_v128_balanced": ["m2rnn_bf16_tc5.cu"],
    "mma_sync_cluster4_k64_v128": ["m2rnn_bf16_cluster.cu"],
    "mma_sync_rows8_cluster8_k64_v128": ["m2rnn_bf16_c8.cu"],
    "mma_sync_rows8_cluster4x2_k64_v128": ["m2rnn_bf16_c8.cu"],
    "mma_sync_rows8": ["m2rnn_bf16_r8.cu"],
    "mma_sync_rows8_cluster2": ["m2rnn_bf16_r8.cu"],
    "backward_mma_k64_v64": ["m2rnn_bwd_bf16_mma.cu"],
    "backward_tc_k64_v64": ["m2rnn_bwd_bf16_tc.cu"],
    "backward_tc8_k64_v64": ["m2rnn_bwd_bf16_tc.cu"],
    "backward_tcc_k64_v64": ["m2rnn_bwd_bf16_tcc.cu"],
    "backward_simt": ["m2rnn_bwd_f32.cu"],
    "backward_tc_v128": ["m2rnn_bwd_bf16_tc128.cu"],
    "backward_tc_v128_t": ["m2rnn_bwd_bf16_tc128t.cu"],
    "decode_bf16_mma": ["m2rnn_decode.cu"],
    "decode_bf16_persist": ["m2rnn_decode.cu"],
    "conv_silu": ["m2rnn_block.cu"],
    "gate_rmsnorm": ["m2rnn_block.cu"],
}


def kernel_source_hash(variant_name):
    """sha256 over the kernel's source file and the shared device helpers."""
    import hashlib
    csrc = os.path.join(ROOT, "matrix_state_nonlinear_gb300", "csrc")
    hsh = hashlib.sha256()
    for f in KERNEL_SOURCES.get(variant_name, []) + ["ptx_util.cuh"]:
        with open(os.path.join(csrc, f), "rb") as fh:
            hsh.update(fh.read())
    return hsh.hexdigest()


def measured_traffic(variant_name, wl):
    """DRAM bytes per launch from the committed ncu capture, scaled to this workload.

    profiles/traffic.json records, per kernel, dram__bytes_read.sum +
    dram__bytes_write.sum of one captured launch, the units (token-heads) that launch
    processed and the source hash of the kernel at capture time.  Traffic grows in
    proportion to the units processed (every input row is read once and every output
    row written once), so it is scaled by units.  Returns None when there is no capture
    or the kernel has changed since it was taken.
    """
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh).get(variant_name)
    if not rec or rec.get("source_sha256") != kernel_source_hash(variant_name):
        return None
    return rec["bytes_per_launch"] * wl.units / rec["units"]


# ---------------------------------------------------------------- replicas across ranks
# The (batch, head) pairs are independent and the recurrence has no exchange step, so
# N GPUs run N replicas of the workload: rank r owns batch rows [r B, (r + 1) B) of a
# global batch N B, drawn with seed r.  The only cross-rank operations are the
# barrier around the timed region and the max of the step times.
def rank_seed(rank: int) -> int:
    return rank


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest `value` over all ranks (the slowest rank sets the job's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job units per second: every rank's units over the slowest rank's time."""
    return world * units_per_rank / (ms_per_step / 1e3)


def pipelined_e2e(dev, stream, warmup, steps, h2d_pairs, compute, d2h_pairs):
    """Milliseconds per end-to-end step with the host copies overlapped, as a serving loop runs.

    Step k copies its inputs from pinned host memory into device set k % 2 on one copy
    stream, runs its kernels on `stream` and copies its results back on another copy stream,
    so step k+1's inputs and step k-1's results move while step k computes.  Events order
    every buffer set's writes after its readers (inputs after the kernels of step k-2, results
    after the copy-out of step k-2).  Every step's own copies are inside the timed region.
    h2d_pairs(i) / d2h_pairs(i) give (device, host) / (host, device) tensor pairs of set i;
    compute(i) launches the step's kernels on `stream`.
    """
    import torch
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    count = [0]

    def run():
        k = count[0]
        i = k % 2
        if k >= 2:
            s_in.wait_event(ev_comp[i])
        with torch.cuda.stream(s_in):
            for d, h in h2d_pairs(i):
                d.copy_(h, non_blocking=True)
        ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        if k >= 2:
            stream.wait_event(ev_out[i])
        compute(i)
        ev_comp[i].record(stream)
        s_out.wait_event(ev_comp[i])
        with torch.cuda.stream(s_out):
            for h, d in d2h_pairs(i):
                h.copy_(d, non_blocking=True)
        ev_out[i].record(s_out)
        count[0] += 1
        return i

    for _ in range(warmup):
        run()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    last = 0
    for _ in range(steps):
        last = run()
    stream.wait_event(ev_out[last])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / steps


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            return json.load(fh), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- clocks sampler
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- CPU oracle sample
def host_cores() -> dict:
    """What the host offers: logical CPUs, and the ones this process may run on."""
    aff = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"host_cpu_count": os.cpu_count(), "affinity_cores": aff}


def _as_f64(x):
    """A worker's input block as fp64: bf16 arrives as its uint16 bit pattern (exact upcast)."""
    import numpy as np
    if x is None:
        return None
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def _oracle_worker(task):
    """One block of (batch, head) pairs through the fp64 oracle, unchanged.  Returns the
    monotonic start and end of the oracle call (system-wide clock) and its CPU seconds."""
    kind, blk = task
    from oracle import m2rnn_backward, m2rnn_forward
    a = {k: _as_f64(v) for k, v in blk.items()}
    c0 = time.process_time()
    t0 = time.monotonic()
    if kind == "forward":
        m2rnn_forward(a["q"], a["k"], a["v"], a["a"], a["alpha"], a["beta"], a["W"], a["w_r"],
                      a["H0"])
    else:                                   # forward keeping states + backward
        m2rnn_backward(a["q"], a["k"], a["v"], a["a"], a["alpha"], a["beta"], a["W"], a["w_r"],
                       a["dy"], a["H0"])
    return t0, time.monotonic(), time.process_time() - c0


def pair_blocks(arrs: dict, parts: int) -> list:
    """Splits a problem's host arrays into at most `parts` blocks of whole (batch, head)
    pairs: heads first, then batch rows.  Pairs are independent units of the recurrence,
    so the blocks' outputs are exactly the full problem's.  Returns a list of
    ((b0, b1, n0, n1), block arrays)."""
    import numpy as np
    B, _, N = arrs["v"].shape[:3]
    gn = max(1, min(N, parts))
    gb = max(1, min(B, parts // gn))
    shared = arrs["q"].shape[2] == 1 and N > 1
    out = []
    for bs in np.array_split(np.arange(B), gb):
        for ns in np.array_split(np.arange(N), gn):
            b0, b1, n0, n1 = int(bs[0]), int(bs[-1]) + 1, int(ns[0]), int(ns[-1]) + 1
            blk = {}
            for key, val in arrs.items():
                if val is None:
                    blk[key] = None
                elif key in ("q", "k"):
                    blk[key] = val[b0:b1, :, :] if shared else val[b0:b1, :, n0:n1]
                elif key in ("v", "a", "dy"):
                    blk[key] = val[b0:b1, :, n0:n1]
                elif key == "H0":
                    blk[key] = val[b0:b1, n0:n1]
                else:                       # alpha, beta, W, w_r: per head
                    blk[key] = val[n0:n1]
                if blk[key] is not None:
                    blk[key] = np.ascontiguousarray(blk[key])
            out.append(((b0, b1, n0, n1), blk))
    return out


class OraclePool:
    """Worker processes (spawned, one BLAS thread each) that run the oracle on blocks of
    independent (batch, head) pairs, one block per core."""

    def __init__(self, procs: int | None = None):
        import multiprocessing as mp
        self.procs = procs or host_cores()["affinity_cores"] or 1
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                                 "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(self.procs)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def run(self, kind: str, arrs: dict):
        """Wall seconds of the parallel oracle run (first start to last end) and CPU seconds."""
        res = self.pool.map(_oracle_worker,
                            [(kind, b) for _, b in pair_blocks(arrs, self.procs)], chunksize=1)
        return max(r[1] for r in res) - min(r[0] for r in res), sum(r[2] for r in res)

    def close(self):
        self.pool.close()
        self.pool.join()


def host_arrays(inp: dict) -> dict:
    """Host copies of the inputs for the oracle workers: bf16 as uint16 bit patterns."""
    import torch
    out = {}
    for k, v in inp.items():
        if v is None:
            out[k] = None
        elif v.dtype == torch.bfloat16:
            out[k] = v.detach().cpu().view(torch.int16).numpy().view("uint16")
        else:
            out[k] = v.detach().cpu().numpy()
    return out


def oracle_sample(wl, seconds: float, T_s: int | None = None, pool: OraclePool | None = None):
    """Times the fp64 oracle on a bounded sample of the workload, on every host core.

    The sample is every (batch, head) pair of the workload over its first T_s
    time steps; without a given T_s it is grown until one run takes about
    `seconds` of wall time.  The pairs are split into one block per core, each run
    by the unchanged oracle in its own process.  Returns (units per second, sample
    description, cores used, T_s).
    """
    from matrix_state_nonlinear_gb300.inputs import make_inputs

    own = pool is None
    pool = pool or OraclePool()
    try:
        fixed = T_s is not None
        T_s = T_s or 8
        while True:
            arrs = host_arrays(make_inputs(wl.with_(T=T_s), "cpu", 0))
            wall, cpu = pool.run("forward", arrs)
            if fixed or wall >= seconds or T_s >= wl.T:
                break
            grow = max(2.0, min(8.0, 1.1 * seconds / max(wall, 1e-3)))
            T_s = min(wl.T, int(T_s * grow))
    finally:
        if own:
            pool.close()
    units = wl.B * wl.N * T_s
    blocks = min(pool.procs, wl.B * wl.N)
    desc = (f"all {wl.B * wl.N} (batch, head) pairs of {wl.name} over the first {T_s} of "
            f"{wl.T} steps (fp64 NumPy oracle, {units} token-heads, {wall:.1f} s wall; pairs "
            f"split into {blocks} blocks run by {pool.procs} single-threaded processes, "
            f"{cpu / wall if wall > 0 else 0:.1f} cores busy on average)")
    return units / wall, desc, blocks, T_s


def reference_arm(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    # Each step is a sample of about `per` seconds of oracle wall time, so that the whole run
    # (warm-up included) stays near two minutes; the sizing below may overshoot by up to 2x.
    per = max(0.25, min(args.cpu_seconds, 60.0 / max(1, args.steps + args.warmup)))
    vals = []
    pool = OraclePool()
    try:
        _, desc, cores, T_s = oracle_sample(wl, per, pool=pool)   # sizes the sample (untimed)
        for i in range(args.warmup + args.steps):
            v, desc, cores, _ = oracle_sample(wl, per, T_s, pool=pool)
            if i >= args.warmup:
                vals.append(v)
    finally:
        pool.close()
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        # The oracle's rate on the sample, carried to the whole workload: the time one full
        # step of this workload would take at that rate.
        "ms_per_step": wl.units / value * 1e3, "ms_per_step_basis": "projected from the sample",
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc, **host_cores()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def input_bytes(wl):
    e = 2 if wl.dtype == "bf16" else 4
    return wl.units * e * (2 * wl.K + wl.V + 1)


def workload_config(wl):
    big = input_bytes(wl) > L2_BYTES
    return {"workload": wl.name, "B": wl.B, "T": wl.T, "N": wl.N, "K": wl.K, "V": wl.V,
            "operands": wl.dtype, "state": "f32",
            "l2": ("inputs larger than L2 (no flush between steps)" if big else
                   "L2 flushed (256 MB write) between steps, outside the timed launches"),
            "parallelism": "replicas (one independent workload per GPU)"}


# ---------------------------------------------------------------- training step
METRIC_TRAIN = "M²RNN training step (state-keeping forward + backward) tokens·heads/s"


def oracle_train_sample(wl, seconds: float, pool: OraclePool | None = None):
    """Times the fp64 oracle's forward + backward on every pair over a bounded prefix of T,
    on every host core (one block of pairs per single-threaded process)."""
    import numpy as np
    from matrix_state_nonlinear_gb300.inputs import make_inputs

    own = pool is None
    pool = pool or OraclePool()
    try:
        T_s = 4
        while True:
            arrs = host_arrays(make_inputs(wl.with_(T=T_s), "cpu", 0))
            arrs["dy"] = np.random.default_rng(1).normal(0, 1, (wl.B, T_s, wl.N, wl.V))
            wall, cpu = pool.run("train", arrs)
            if wall >= seconds or T_s >= wl.T:
                break
            T_s = min(wl.T, int(T_s * max(2.0, min(8.0, 1.1 * seconds / max(wall, 1e-3)))))
    finally:
        if own:
            pool.close()
    units = wl.B * wl.N * T_s
    blocks = min(pool.procs, wl.B * wl.N)
    desc = (f"all {wl.B * wl.N} (batch, head) pairs of {wl.name} over the first {T_s} of "
            f"{wl.T} steps (fp64 NumPy oracle, forward keeping states + backward, {units} "
            f"token-heads, {wall:.1f} s wall; pairs split into {blocks} blocks run by "
            f"{pool.procs} single-threaded processes, {cpu / wall if wall > 0 else 0:.1f} cores "
            f"busy on average)")
    return units / wall, desc, blocks


def main_train(args, wl):
    """One step = m2rnn_forward_train (y, H_T and every state H_t) + m2rnn_backward
    (all gradients) over the workload, with a fixed synthetic upstream gradient dy."""
    import torch
    import torch.distributed as dist

    import __graft_entry__
    import matrix_state_nonlinear_gb300 as pkg
    from matrix_state_nonlinear_gb300.inputs import make_inputs

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    pkg.load_library()

    inp = make_inputs(wl, dev, seed=rank_seed(rank))
    B, T, N, K, V = wl.B, wl.T, wl.N, wl.K, wl.V
    Nqk = 1 if wl.shared_qk else N
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + rank)
    dy = torch.randn((B, T, N, V), generator=g, device=dev)
    y = torch.empty((B, T, N, V), dtype=torch.float32, device=dev)
    HT = torch.empty((B, N, K, V), dtype=torch.float32, device=dev)
    Hs = torch.empty((B, N, T, K, V), dtype=torch.bfloat16 if wl.dtype == "bf16" else torch.float32,
                     device=dev)
    grads = {"dq": (B, T, Nqk, K), "dk": (B, T, Nqk, K), "dv": (B, T, N, V), "da": (B, T, N),
             "dalpha": (N,), "dbeta": (N,), "dW": (N, V, V), "dw_r": (N, V), "dH0": (B, N, K, V)}
    grads = {n: torch.empty(shp, dtype=torch.float32, device=dev) for n, shp in grads.items()}
    ws = torch.empty(max(16, pkg.backward_workspace_bytes(B, T, N, Nqk, K, V)), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream(dev)
    marks = []

    def step(record=False):
        if record:
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record(stream)
        pkg.m2rnn_forward_train(inp, y=y, H_T=HT, Hs=Hs, stream=stream)
        if record:
            e[1].record(stream)
        pkg.m2rnn_backward(inp, Hs, dy, grads=grads, workspace=ws, variant=args.variant,
                           stream=stream)
        if record:
            e[2].record(stream)
            marks.append(e)

    for _ in range(args.warmup):
        step()
    if pkg.stream_status(stream) != 0:
        raise RuntimeError("device status not OK after warm-up")
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step(record=True)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    total_ms = ev0.elapsed_time(ev1)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    if pkg.stream_status(stream) != 0:
        raise RuntimeError("device status not OK after the timed steps")
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in marks)
    bwd_ms = statistics.mean(b.elapsed_time(c) for _, b, c in marks)
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(wl.units, world, ms_per_step)

    e2e = None
    if not args.no_e2e:
        names = ["q", "k", "v", "a", "alpha", "beta", "W", "w_r", "H0"]
        host = {k: inp[k].cpu().pin_memory() for k in names if inp.get(k) is not None}
        dinp = {k: torch.empty_like(inp[k]) for k in host}
        if "H0" not in dinp:
            dinp["H0"] = None
        dy_h = dy.cpu().pin_memory()
        dy_d = torch.empty_like(dy)
        out_h = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in grads.items()}
        h2d = sum(v.numel() * v.element_size() for v in host.values()) + dy_h.numel() * 4
        d2h = sum(t.numel() * 4 for t in out_h.values())

        def e2e_step():
            for k, v in host.items():
                dinp[k].copy_(v, non_blocking=True)
            dy_d.copy_(dy_h, non_blocking=True)
            pkg.m2rnn_forward_train(dinp, y=y, H_T=HT, Hs=Hs, stream=stream)
            pkg.m2rnn_backward(dinp, Hs, dy_d, grads=grads, workspace=ws, variant=args.variant,
                               stream=stream)
            for n, t in grads.items():
                out_h[n].copy_(t, non_blocking=True)

        e_steps = max(3, min(args.steps, 5))
        e2e_step()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        serial_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, world, dev)

        # Overlapped copies: inputs, dy and gradients double-buffered; the kernels of
        # consecutive steps stay in order on `stream`, so Hs and the workspace are shared.
        sets = [dict(dinp), {k: (None if v is None else torch.empty_like(v)) for k, v in dinp.items()}]
        dys = [dy_d, torch.empty_like(dy_d)]
        gsets = [grads, {n: torch.empty_like(t) for n, t in grads.items()}]
        gh = [out_h, {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                      for n, t in grads.items()}]

        def train_compute(i):
            pkg.m2rnn_forward_train(sets[i], y=y, H_T=HT, Hs=Hs, stream=stream)
            pkg.m2rnn_backward(sets[i], Hs, dys[i], grads=gsets[i], workspace=ws,
                               variant=args.variant, stream=stream)

        p_steps = max(5, min(args.steps, 10))
        e_ms = max_over_ranks(pipelined_e2e(
            dev, stream, 1, p_steps,
            lambda i: [(sets[i][k], v) for k, v in host.items()] + [(dys[i], dy_h)],
            train_compute,
            lambda i: [(gh[i][n], gsets[i][n]) for n in gsets[i]]), world, dev)
        e2e = {"value": job_throughput(wl.units, world, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "steps": p_steps, "serial_ms_per_step": serial_ms, "serial_steps": e_steps,
               "overlap": "step k+1's host-to-device and step k-1's device-to-host copies run on "
                          "two copy streams during step k's kernels (double-buffered device "
                          "sets); serial_ms_per_step: the same steps on one stream"}

    # ---- roofline of the dominant kernel: the backward's reverse scan
    peaks, peak_src = load_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    flops = 6.0 * K * V * V * wl.units   # H_{t-1} W (recomputed), D_t W^T, H_{t-1}^T D_t
    e = 2 if wl.dtype == "bf16" else 4   # operand bytes; the kept states use the same dtype
    bwd_bytes = wl.units * (e * K * V + 4 * V + e * (2 * K + V + 1) + 4 * (2 * K + V + 1))
    fwd_bytes = wl.units * (e * K * V + e * (2 * K + V + 1) + 4 * V)
    achieved = flops / (bwd_ms / 1e3) / 1e12
    mma = wl.dtype == "bf16" and K == 64 and V == 64 and args.variant in (0, 2, 3, 4, 5)
    v128 = wl.dtype == "bf16" and V == 128 and K % 16 == 0 and args.variant in (0, 6, 7)
    # V = 128: the products transposed for K <= 64 (variant 7, the automatic choice there)
    v128t = v128 and (args.variant == 7 or (args.variant == 0 and K <= 64))
    if mma or v128:   # bf16 tensor-core products: the measured bf16 dense peak
        peak, bound = float(peaks["bf16_tflops"]), "tensor"
        psrc = f"{peak_src} bf16 dense burst (kernel timed alone)"
        kname = ("backward_tc_v128_t" if v128t else "backward_tc_v128") if v128 else {
            2: "backward_mma_k64_v64", 4: "backward_tc8_k64_v64",
            3: "backward_tc_k64_v64"}.get(args.variant, "backward_tcc_k64_v64")
    else:     # fp32 SIMT arithmetic: SMs x 128 FMA lanes x 2 flop x max SM clock
        max_mhz = clk.get("sm_max_mhz") or 2070.0
        peak, bound = sms * 128 * 2 * max_mhz * 1e6 / 1e12, "alu"
        psrc, kname = "fp32 FMA peak from unit counts and the maximum SM clock", "backward_simt"
    roof = {"bound": bound, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "peak_source": psrc,
            "kernel": kname, "traffic": measured_traffic(kname, wl),
            "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": bwd_bytes,
            "hbm_frac": bwd_bytes / (bwd_ms / 1e3) / 1e9 / float(peaks["hbm_gbs"]),
            "backward_ms": bwd_ms, "forward_train_ms": fwd_ms,
            "forward_train_hbm_frac": fwd_bytes / (fwd_ms / 1e3) / 1e9 / float(peaks["hbm_gbs"]),
            "t_hbm_roofline_ms": (fwd_bytes + bwd_bytes) / (float(peaks["hbm_gbs"]) * 1e9) * 1e3,
            "hbm_peak_gbs": float(peaks["hbm_gbs"]), "hbm_peak_source": peak_src}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, desc, cores = oracle_train_sample(wl, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
               **host_cores()}
    launches = 2 + (1 if Nqk == 1 and N > 1 else 0) + 1    # forward, backward, reduce(s)
    if rank == 0:
        line = {"metric": METRIC_TRAIN, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if wl.dtype == "bf16" else "f32", "data": "synthetic",
                "config": dict(workload_config(wl), **{"pass": "train"}), "clocks": clk,
                "e2e": e2e, "gpu_launches": args.steps * launches, "roofline": roof,
                "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------- decode step
METRIC_DECODE = "M²RNN decode step (T = 1, state in / out) tokens·heads/s"
# Serving batches for the headline head shape (N = 16, K = V = 64).  The large batch
# keeps 268 MB of fp32 state, more than L2, so each step streams the state from HBM.
DECODE_BATCHES = {"decode_b1024_n16_k64_v64": 1024, "decode_b8_n16_k64_v64": 8}


def decode_reference(args):
    """The fp64 oracle on the same decode step (one token, the whole batch)."""
    rank, _, _ = dist_env()
    if rank != 0:
        return 0
    from matrix_state_nonlinear_gb300.inputs import Workload, make_inputs, to_f64_numpy
    from oracle import m2rnn_forward

    name = args.workload if args.workload in DECODE_BATCHES else "decode_b1024_n16_k64_v64"
    B, N, K, V = DECODE_BATCHES[name], 16, 64, 64
    arrs = {k: to_f64_numpy(v) for k, v in
            make_inputs(Workload(name, B, 1, N, K, V, h0="uniform"), "cpu", 0).items()}
    vals = []
    c0, t_all = time.process_time(), time.perf_counter()
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        m2rnn_forward(arrs["q"], arrs["k"], arrs["v"], arrs["a"], arrs["alpha"], arrs["beta"],
                      arrs["W"], arrs["w_r"], arrs["H0"])
        if i >= args.warmup:
            vals.append(B * N / (time.perf_counter() - t0))
    cores = max(1, round((time.process_time() - c0) / (time.perf_counter() - t_all)))
    value = statistics.median(vals)
    desc = (f"one decode step of {name} (fp64 NumPy oracle, {B * N} token-heads per step; "
            f"one process: a decode step is too short to split across cores)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC_DECODE, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": None,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": name, "B": B, "T": 1, "N": N, "K": K, "V": V,
                                        "pass": "decode"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc, **host_cores()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)
    return 0


def main_decode(args):
    """One step = one m2rnn_decode_step_bf16 call over the batch (state updated in place).
    Also reports the per-step latency with the steps replayed from a CUDA graph."""
    import torch

    import __graft_entry__
    import matrix_state_nonlinear_gb300 as pkg
    from matrix_state_nonlinear_gb300.inputs import Workload, make_inputs

    name = args.workload if args.workload in DECODE_BATCHES else "decode_b1024_n16_k64_v64"
    B, N, K, V = DECODE_BATCHES[name], 16, 64, 64
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    __graft_entry__.build()
    pkg.load_library()
    wl = Workload(name, B, 1, N, K, V, h0="uniform")
    inp = make_inputs(wl, dev, seed=rank_seed(rank))
    args_ = (inp["q"][:, 0].contiguous(), inp["k"][:, 0].contiguous(), inp["v"][:, 0].contiguous(),
             inp["a"][:, 0].contiguous(), inp["alpha"], inp["beta"], inp["W"], inp["w_r"])
    H = inp["H0"].clone()
    y = torch.empty((B, N, V), device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        pkg.m2rnn_decode_step(*args_, H, y=y, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    if pkg.stream_status(stream) != 0:
        raise RuntimeError("device status not OK after warm-up")
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    ms = ev0.elapsed_time(ev1) / args.steps
    # the same steps replayed from a CUDA graph (no per-call host work)
    g_steps = 64
    s2 = torch.cuda.Stream(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s2):
        with torch.cuda.graph(graph, stream=s2):
            for _ in range(g_steps):
                pkg.m2rnn_decode_step(*args_, H, y=y, stream=s2)
    graph.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    graph_ms = e0.elapsed_time(e1) / g_steps
    clk = clocks.stop()
    if pkg.stream_status(stream) != 0:
        raise RuntimeError("device status not OK after the timed steps")
    units = B * N
    value = units / (ms / 1e3)

    e2e = None
    if not args.no_e2e:
        names = ["q", "k", "v", "a"]
        host = [x.cpu().pin_memory() for x in args_[:4]]
        dev_in = [torch.empty_like(x) for x in args_[:4]]
        y_h = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
        h2d = sum(x.numel() * x.element_size() for x in host)
        d2h = y_h.numel() * 4

        def e2e_step():
            for d, h in zip(dev_in, host):
                d.copy_(h, non_blocking=True)
            pkg.m2rnn_decode_step(*dev_in, *args_[4:], H, y=y, stream=stream)
            y_h.copy_(y, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(dev)
        e_steps = max(10, min(args.steps, 200))
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(e_steps):
            e2e_step()
        a1.record(stream)
        torch.cuda.synchronize(dev)
        serial_ms = a0.elapsed_time(a1) / e_steps
        # Overlapped: the next token's inputs and the previous token's y move on copy
        # streams while this token's step runs (the state stays resident and in order).
        din = [dev_in, [torch.empty_like(x) for x in dev_in]]
        ys = [y, torch.empty_like(y)]
        yh = [y_h, torch.empty(y.shape, dtype=y.dtype, pin_memory=True)]
        e_ms = pipelined_e2e(
            dev, stream, 2, e_steps, lambda i: list(zip(din[i], host)),
            lambda i: pkg.m2rnn_decode_step(*din[i], *args_[4:], H, y=ys[i], stream=stream),
            lambda i: [(yh[i], ys[i])])
        e2e = {"value": units / (e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms, "steps": e_steps,
               "serial_ms_per_step": serial_ms,
               "note": "token inputs host->device, y device->host; the state stays resident. "
                       "ms_per_step overlaps the next token's input copy and the previous "
                       "token's y copy with this token's step (double-buffered); "
                       "serial_ms_per_step: the same steps on one stream"}

    peaks, peak_src = load_peaks()
    # K = V = 64 with at least 2048 (batch, head) pairs runs the persistent TMA-fed kernel
    kname = "decode_bf16_persist" if B * N >= 2048 else "decode_bf16_mma"
    hbm = units * (2 * K * V * 4 + 2 * (2 * K + V + 1) + 4 * V) + N * V * V * 2
    achieved = hbm / (ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
            "frac": achieved / float(peaks["hbm_gbs"]),
            "peak_source": f"{peak_src} HBM copy bandwidth", "kernel": kname,
            "traffic": measured_traffic(kname, wl),
            "algorithmic_bytes_per_launch": hbm, "graph_replay_ms_per_step": graph_ms,
            "graph_achieved_gbs": hbm / (graph_ms / 1e3) / 1e9}
    line = {"metric": METRIC_DECODE, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": name, "B": B, "T": 1, "N": N, "K": K, "V": V,
                       "operands": "bf16", "state": "f32", "pass": "decode",
                       "l2": ("state larger than L2 (no flush between steps)" if
                              B * N * K * V * 4 > L2_BYTES else
                              "state fits in L2 (latency case; not flushed)"),
                       "parallelism": "replicas (one independent workload per GPU)"},
            "clocks": clk, "e2e": e2e, "gpu_launches": args.steps, "roofline": roof,
            "cpu_baseline": None}
    if not args.no_cpu_baseline:   # the oracle on the same step, on the host cores
        from matrix_state_nonlinear_gb300.inputs import to_f64_numpy
        from oracle import m2rnn_forward
        Bs = max(1, min(B, 256))   # a bounded sample of the batch
        arrs = {k_: to_f64_numpy(v_[:Bs] if k_ in ("q", "k", "v", "a", "H0") else v_)
                for k_, v_ in inp.items()}
        c0, t0 = time.process_time(), time.perf_counter()
        m2rnn_forward(arrs["q"], arrs["k"], arrs["v"], arrs["a"], arrs["alpha"], arrs["beta"],
                      arrs["W"], arrs["w_r"], arrs["H0"])
        wall = time.perf_counter() - t0
        line["cpu_baseline"] = {
            "value": Bs * N / wall, "unit": UNIT, "kind": "oracle",
            "cores": max(1, round((time.process_time() - c0) / wall)), **host_cores(),
            "sample": f"one decode step of the first {Bs} of {B} batch rows "
                      f"(fp64 NumPy oracle, {Bs * N} token-heads, {wall:.2f} s wall; one "
                      f"process)"}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- block (prologue + forward + epilogue)
METRIC_BLOCK = ("M²RNN block recurrence path (conv/SiLU on q, k, v + forward + gate/RMSNorm) "
                "tokens·heads/s")


def main_block(args, wl):
    """One step = the conv/SiLU prologue on the q, k, v projections, the forward recurrence,
    and m2rnn_gate_rmsnorm_bf16 on its readout (the GEMM projections are not included).
    The step is the three-stage chain (m2rnn_conv_silu_bf16 per projection, forward,
    epilogue); where the eight-row kernels take the shape, the fused entry
    (m2rnn_forward_conv_bf16: prologue inside the forward) plus the epilogue is timed too and
    reported beside it (it is slower: the forward is bound by per-step issue on each
    sub-partition, which the prologue's work joins)."""
    import torch

    import __graft_entry__
    import matrix_state_nonlinear_gb300 as pkg
    from matrix_state_nonlinear_gb300.inputs import make_inputs

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    __graft_entry__.build()
    pkg.load_library()
    if wl.dtype != "bf16":
        raise SystemExit("--pass block runs the bf16 path")
    inp = make_inputs(wl, dev, seed=rank_seed(rank))
    B, T, N, K, V = wl.B, wl.T, wl.N, wl.K, wl.V
    Nqk = 1 if wl.shared_qk else N
    g = torch.Generator(device=dev)
    g.manual_seed(2000 + rank)
    pre = {n: torch.randn((B, T, c), generator=g, device=dev).to(torch.bfloat16)
           for n, c in (("q", Nqk * K), ("k", Nqk * K), ("v", N * V))}
    cw = {n: 0.5 * torch.randn((x.shape[2], 4), generator=g, device=dev) for n, x in pre.items()}
    conv = {"w" + n: cw[n] for n in cw}
    fused_in = dict(inp)
    for n in ("q", "k", "v"):
        fused_in[n] = pre[n].view(B, T, -1, K if n != "v" else V)
    fused = K in (32, 64) and V in (16, 32, 48, 64)
    gpre = torch.randn((B, T, N * V), generator=g, device=dev).to(torch.bfloat16)
    wn = 1.0 + 0.1 * torch.randn(N * V, generator=g, device=dev)
    run = dict(inp)
    for n in ("q", "k", "v"):
        run[n] = torch.empty_like(pre[n]).view(B, T, -1, K if n != "v" else V)
    y = torch.empty((B, T, N, V), device=dev)
    HT = torch.empty((B, N, K, V), device=dev)
    out = torch.empty((B, T, N * V), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    marks = []

    fused_marks = []

    def fused_step(record=False):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)] if record else None
        if record:
            e[0].record(stream)
        pkg.m2rnn_forward_conv(fused_in, conv, y=y, H_T=HT, stream=stream)
        if record:
            e[1].record(stream)
        pkg.gate_rmsnorm(y.view(B, T, N * V), gpre, wn, 1e-6, out=out, stream=stream)
        if record:
            e[2].record(stream)
            fused_marks.append(e)

    def step(record=False):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)] if record else None
        if record:
            e[0].record(stream)
        for n in ("q", "k", "v"):
            pkg.conv_silu(pre[n], cw[n], out=run[n].view(B, T, -1), stream=stream)
        if record:
            e[1].record(stream)
        pkg.m2rnn_forward(run, y=y, H_T=HT, stream=stream)
        if record:
            e[2].record(stream)
        pkg.gate_rmsnorm(y.view(B, T, N * V), gpre, wn, 1e-6, out=out, stream=stream)
        if record:
            e[3].record(stream)
            marks.append(e)

    for _ in range(max(3, args.warmup)):
        step()
        if fused:
            fused_step()
    if pkg.stream_status(stream) != 0:
        raise RuntimeError("device status not OK after warm-up")
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)

    def timed(fn):
        torch.cuda.synchronize(dev)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            fn(record=True)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        return ev0.elapsed_time(ev1) / args.steps

    unfused_ms = timed(step)
    fused_ms = timed(fused_step) if fused else None
    clk = clocks.stop()
    if pkg.stream_status(stream) != 0:
        raise RuntimeError("device status not OK after the timed steps")
    ms = unfused_ms
    pro_ms = statistics.mean(a.elapsed_time(b) for a, b, _, _ in marks)
    fwd_ms = statistics.mean(b.elapsed_time(c) for _, b, c, _ in marks)
    epi_ms = statistics.mean(c.elapsed_time(d) for _, _, c, d in marks)
    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    pro_bytes = sum(x.numel() for x in pre.values()) * 4          # bf16 in + bf16 out
    epi_bytes = B * T * N * V * (4 + 2 + 2)                        # y f32, g bf16 in; out bf16
    flops = 2.0 * K * V * V * wl.units
    peak_t = float(peaks["bf16_tflops"])
    roof = {"bound": "tensor", "achieved": flops / (fwd_ms / 1e3) / 1e12, "peak": peak_t,
            "unit": "TFLOP/s", "frac": flops / (fwd_ms / 1e3) / 1e12 / peak_t,
            "peak_source": f"{peak_src} bf16 dense burst (kernel timed alone)",
            "kernel": pkg.variant_name(pkg.pick_variant(B, T, N, K, V)),
            "traffic": measured_traffic(pkg.variant_name(pkg.pick_variant(B, T, N, K, V)), wl),
            "forward_ms": fwd_ms, "prologue_ms": pro_ms, "epilogue_ms": epi_ms,
            "prologue_hbm_frac": pro_bytes / (pro_ms / 1e3) / 1e9 / hbm,
            "epilogue_hbm_frac": epi_bytes / (epi_ms / 1e3) / 1e9 / hbm,
            "prologue_bytes": pro_bytes, "epilogue_bytes": epi_bytes,
            "hbm_peak_gbs": hbm, "unfused_ms_per_step": unfused_ms,
            "fused_ms_per_step": fused_ms,
            "fused_forward_ms": (statistics.mean(a.elapsed_time(b) for a, b, _ in fused_marks)
                                 if fused else None),
            "step": "prologue, forward, epilogue as three stages"}
    line = {"metric": METRIC_BLOCK, "value": wl.units / (ms / 1e3), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": dict(workload_config(wl), **{"pass": "block"}),
            "clocks": clk, "e2e": None, "gpu_launches": args.steps * 5,
            "roofline": roof,
            "cpu_baseline": None}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm
def serial_bound(pkg, inp, wl, variant, stream, dev, ms_per_step, mhz, T_s=4096):
    """The serial-latency bound of T dependent steps, measured with the library's kernels.

    One (batch, head) pair alone on the GPU (B = N = 1, its first T_s steps) runs the
    dependent step chain with nothing else competing for its SM(s).  Two forms are timed:
    the workload's own variant on one pair (`serial_same_variant`), and the variant the
    library picks for a lone pair (at K = V = 64 the pair split over a two-block cluster,
    one compute warp per sub-partition).  The faster one's per-step time times T is the
    least time these kernels take for T steps of one pair; when the workload has no more
    pairs than the GPU runs at once, the whole job is bound by this chain."""
    import torch
    T_s = min(wl.T, T_s)
    one = {}
    for k, v in inp.items():
        if v is None:
            one[k] = None
        elif k in ("q", "k", "v", "a"):
            one[k] = v[0:1, :T_s, 0:1].contiguous()
        elif k == "H0":
            one[k] = v[0:1, 0:1].contiguous()
        else:
            one[k] = v[0:1].contiguous()
    y1 = torch.empty((1, T_s, 1, wl.V), dtype=torch.float32, device=dev)
    H1 = torch.empty((1, 1, wl.K, wl.V), dtype=torch.float32, device=dev)
    own = variant or pkg.pick_variant(wl.B, wl.T, wl.N, wl.K, wl.V)
    lone = pkg.pick_variant(1, T_s, 1, wl.K, wl.V)

    def per_step_ms(v):
        for _ in range(2):
            pkg.m2rnn_forward(one, y=y1, H_T=H1, variant=v, stream=stream)
        times = []
        for _ in range(5):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            pkg.m2rnn_forward(one, y=y1, H_T=H1, variant=v, stream=stream)
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        return statistics.median(times) / T_s

    def cycles(ms):
        return ms * 1e-3 * mhz * 1e6

    own_ms = per_step_ms(own)
    lone_ms = own_ms if lone == own else per_step_ms(lone)
    best_ms, best_v = (lone_ms, lone) if lone_ms < own_ms else (own_ms, own)
    t_serial = best_ms * wl.T
    return {"t_serial_bound_ms": t_serial,
            "serial_cycles_per_step": cycles(best_ms),
            "serial_frac": t_serial / ms_per_step,
            "serial_variant": pkg.variant_name(best_v),
            "serial_same_variant": {"variant": pkg.variant_name(own),
                                    "cycles_per_step": cycles(own_ms),
                                    "t_ms": own_ms * wl.T},
            "serial_method": (f"one (batch, head) pair alone (B = N = 1, first {T_s} steps, "
                              f"median of 5 CUDA-event-timed launches) on the workload's "
                              f"variant and on the variant picked for a lone pair; the faster "
                              f"per-step time x T; cycles at the median sampled SM clock")}


def main():
    args = parse()
    from matrix_state_nonlinear_gb300.inputs import HEADLINE, WORKLOADS
    if args.which == "decode":
        return main_decode(args) if args.impl == "ours" else decode_reference(args)
    wl = WORKLOADS[args.workload or HEADLINE]
    if args.batch:
        wl = wl.with_(B=args.batch, name=f"{wl.name}_b{args.batch}")
    if args.seq:
        wl = wl.with_(T=args.seq, name=f"{wl.name}_t{args.seq}")
    if args.heads:
        wl = wl.with_(N=args.heads, name=f"{wl.name}_n{args.heads}")
    if args.impl == "reference":
        return reference_arm(args, wl)
    if args.which == "train":
        return main_train(args, wl)
    if args.which == "block":
        return main_block(args, wl)

    import torch
    import torch.distributed as dist

    import __graft_entry__
    import matrix_state_nonlinear_gb300 as pkg
    from matrix_state_nonlinear_gb300.inputs import make_inputs

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    pkg.load_library()

    inp = make_inputs(wl, dev, seed=rank_seed(rank))
    B, T, N, K, V = wl.B, wl.T, wl.N, wl.K, wl.V
    y = torch.empty((B, T, N, V), dtype=torch.float32, device=dev)
    HT = torch.empty((B, N, K, V), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = None if input_bytes(wl) > L2_BYTES else torch.empty(64 << 20, dtype=torch.float32,
                                                                  device=dev)

    def step():
        pkg.m2rnn_forward(inp, y=y, H_T=HT, variant=args.variant, stream=stream)

    for _ in range(args.warmup):
        step()
    if pkg.stream_status(stream) != 0:
        raise RuntimeError("device status not OK after warm-up")

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if flush is None:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        total_ms = ev0.elapsed_time(ev1)
    else:                                   # small inputs: flush L2 between timed launches
        evs = []
        for _ in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step()
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        total_ms = sum(a.elapsed_time(b) for a, b in evs)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    if pkg.stream_status(stream) != 0:
        raise RuntimeError("device status not OK after the timed steps")
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(wl.units, world, ms_per_step)

    # ---- end to end: pinned host inputs -> device -> kernel -> y, H_T back to pinned host
    e2e = None
    if not args.no_e2e:
        host = {k: (None if v is None else v.cpu().pin_memory()) for k, v in inp.items()}
        dinp = {k: (None if v is None else torch.empty_like(v)) for k, v in inp.items()}
        y_h = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
        HT_h = torch.empty(HT.shape, dtype=HT.dtype, pin_memory=True)
        h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
        d2h = y_h.numel() * 4 + HT_h.numel() * 4

        def e2e_step():
            for k, v in host.items():
                if v is not None:
                    dinp[k].copy_(v, non_blocking=True)
            pkg.m2rnn_forward(dinp, y=y, H_T=HT, variant=args.variant, stream=stream)
            y_h.copy_(y, non_blocking=True)
            HT_h.copy_(HT, non_blocking=True)

        e_steps = max(3, min(args.steps, 10))
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        serial_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, world, dev)

        # The same steps with the copies overlapped (two device buffer sets, copy streams).
        sets = [dinp, {k: (None if v is None else torch.empty_like(v)) for k, v in inp.items()}]
        outs = [(y, HT), (torch.empty_like(y), torch.empty_like(HT))]
        outs_h = [(y_h, HT_h), (torch.empty(y.shape, dtype=y.dtype, pin_memory=True),
                                torch.empty(HT.shape, dtype=HT.dtype, pin_memory=True))]
        p_steps = max(10, min(args.steps, 30))  # fill and drain amortised as in a serving loop
        e_ms = max_over_ranks(pipelined_e2e(
            dev, stream, 2, p_steps,
            lambda i: [(sets[i][k], v) for k, v in host.items() if v is not None],
            lambda i: pkg.m2rnn_forward(sets[i], y=outs[i][0], H_T=outs[i][1],
                                        variant=args.variant, stream=stream),
            lambda i: [(outs_h[i][0], outs[i][0]), (outs_h[i][1], outs[i][1])]), world, dev)
        e2e = {"value": job_throughput(wl.units, world, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "steps": p_steps, "serial_ms_per_step": serial_ms, "serial_steps": e_steps,
               "overlap": "step k+1's host-to-device and step k-1's device-to-host copies run on "
                          "two copy streams during step k's kernel (double-buffered device "
                          "sets); serial_ms_per_step: the same steps on one stream"}

    # ---- roofline of the forward kernel (one launch per step)
    peaks, peak_src = load_peaks()
    flops = 2.0 * K * V * V * wl.units
    hbm_bytes = (wl.units * (2 * (2 * K + V + 1) + 4 * V) + N * V * V * 2
                 + (2 if wl.h0 != "zero" else 1) * B * N * K * V * 4)
    launch_s = ms_per_step / 1e3
    tflops = flops / launch_s / 1e12
    peak_t = float(peaks["bf16_tflops"])
    roof = {"bound": "tensor", "achieved": tflops, "peak": peak_t, "unit": "TFLOP/s",
            "frac": tflops / peak_t,
            "peak_source": f"{peak_src} bf16 dense burst (kernel timed alone)",
            "kernel": pkg.variant_name(pkg.pick_variant(B, T, N, K, V) if args.variant == 0
                                       else args.variant),
            "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": hbm_bytes,
            "hbm_frac": hbm_bytes / launch_s / 1e9 / float(peaks["hbm_gbs"]),
            "t_mma_roofline_ms": flops / (peak_t * 1e12) * 1e3,
            "t_hbm_roofline_ms": hbm_bytes / (float(peaks["hbm_gbs"]) * 1e9) * 1e3}
    roof["traffic"] = measured_traffic(roof["kernel"], wl)
    # The MUFU tanh floor: K*V tanh per token-head at 16 per clock per SM (measured rate).
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clk.get("sm_mhz") or 1950.0
    roof["t_mufu_tanh_floor_ms"] = K * V * wl.units / (16.0 * sms * mhz * 1e6) * 1e3
    # The FP32 ALU floor: about four FP32 operations per state element and step (the rank-1
    # product, the gate lerp's multiply and fused multiply-add, the bf16 pack) at 128 lanes
    # per clock per SM.
    roof["t_fp32_alu_floor_ms"] = 4.0 * K * V * wl.units / (128.0 * sms * mhz * 1e6) * 1e3
    roof.update(serial_bound(pkg, inp, wl, args.variant, stream, dev, ms_per_step, mhz))

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, desc, cores, _ = oracle_sample(wl, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
               **host_cores()}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if wl.dtype == "bf16" else "f32", "data": "synthetic",
                "config": workload_config(wl), "clocks": clk, "e2e": e2e,
                "gpu_launches": args.steps, "roofline": roof, "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
