"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Tolerances (max abs error over every element of y and H_T):
  * fp32-operand path: 1e-4;
  * bf16-operand / fp32-state path: 3e-2.
Both sides receive the same seeded inputs (bf16 values upcast exactly to fp64
for the oracle).  Full-size workloads are checked on sampled (batch, head)
pairs, each computed by the oracle in full (every t, every row): pairs are
independent units of the recurrence, so a pair's outputs do not depend on the
others.
"""
import math

import numpy as np
import pytest
import torch

import __graft_entry__
import matrix_state_nonlinear_gb300 as pkg
from matrix_state_nonlinear_gb300 import m2rnn as binding
from matrix_state_nonlinear_gb300.inputs import (WORKLOADS, Workload, all_f64, make_inputs,
                                                 slice_pair)
from oracle import m2rnn_forward_inputs

pytestmark = pytest.mark.gpu
TOL_F32 = 1e-4
TOL_BF16 = 3e-2
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    __graft_entry__.build()
    pkg.load_library()


def run_gpu(inp, variant=0, H_T=True):
    q = inp["q"]
    B, T, _, K = q.shape                     # q may hold one head shared by all
    N, V = inp["v"].shape[2], inp["v"].shape[3]
    y = torch.full((B, T, N, V), float("nan"), device=q.device)
    if H_T:
        HT = torch.full((B, N, K, V), float("nan"), device=q.device)
        pkg.m2rnn_forward(inp, y=y, H_T=HT, variant=variant)
    else:                                    # H_T = NULL through the C ABI
        HT = None
        args = [inp[x] for x in ("q", "k", "v", "a", "alpha", "beta", "W", "w_r")]
        if q.dtype == torch.float32:
            pkg.m2rnn_forward_f32(*args, inp.get("H0"), y, None)
        else:
            pkg.m2rnn_forward_bf16_variant(*args, inp.get("H0"), y, None, variant=variant)
    assert pkg.stream_status() == binding.OK
    return y, HT


def max_err(gpu, ref):
    return float(np.abs(gpu.double().cpu().numpy() - ref).max()) if ref.size else 0.0


def check_full(wl, tol, variant=0, seed=0):
    inp = make_inputs(wl, DEV, seed)
    y, HT = run_gpu(inp, variant)
    yo, HTo = m2rnn_forward_inputs(all_f64(inp))
    ey, eh = max_err(y, yo), max_err(HT, HTo)
    assert ey <= tol and eh <= tol, f"{wl} y err {ey:.3e} H_T err {eh:.3e}"
    return ey, eh


# ---------------------------------------------------------------- fp32 path
def test_f32_tiny_workload_and_golden():
    import json, os
    check_full(WORKLOADS["tiny_f32_b1_t64_n2_k8_v8"], TOL_F32)
    doc = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                      "tiny_f32_b1_t64_n2_k8_v8.json")))
    s, i = doc["shape"], doc["inputs"]
    B, T, N, K, V = s["B"], s["T"], s["N"], s["K"], s["V"]
    t = lambda key, shp: torch.tensor(i[key], dtype=torch.float32, device=DEV).reshape(shp)
    inp = dict(q=t("q", (B, T, N, K)), k=t("k", (B, T, N, K)), v=t("v", (B, T, N, V)),
               a=t("a", (B, T, N)), alpha=t("alpha", (N,)), beta=t("beta", (N,)),
               W=t("W", (N, V, V)), w_r=t("w_r", (N, V)), H0=None)
    y, HT = run_gpu(inp)
    assert max_err(y, np.array(doc["y"]).reshape(B, T, N, V)) <= TOL_F32
    assert max_err(HT, np.array(doc["H_T"]).reshape(B, N, K, V)) <= TOL_F32


F32_SHAPES = [(1, 1, 1, 1, 1), (2, 5, 3, 3, 7), (1, 33, 2, 16, 16), (3, 17, 1, 33, 9),
              (1, 40, 2, 64, 64), (1, 9, 1, 128, 128), (2, 3, 2, 128, 5)]


@pytest.mark.parametrize("B,T,N,K,V", F32_SHAPES)
@pytest.mark.parametrize("h0", ["zero", "uniform"])
def test_f32_shapes(B, T, N, K, V, h0):
    wl = Workload("f32", B, T, N, K, V, dtype="f32", rescale_w=False, h0=h0)
    check_full(wl, TOL_F32, seed=B * 7 + T)


# ---------------------------------------------------------------- bf16 path
BF16_SHAPES = [(1, 1, 1, 16, 16), (1, 2, 1, 16, 32), (3, 17, 1, 16, 64), (1, 63, 3, 32, 16),
               (2, 64, 1, 64, 64), (1, 65, 3, 64, 64), (1, 130, 2, 48, 32), (2, 97, 1, 128, 64),
               (1, 70, 2, 64, 128), (1, 33, 3, 128, 128), (2, 200, 1, 112, 128),
               (1, 1, 1, 64, 128), (1, 129, 1, 64, 128), (2, 300, 3, 64, 128),
               # K a multiple of 8 (eight-row warps), V = 48
               (1, 70, 2, 8, 16), (2, 65, 1, 24, 48), (1, 100, 3, 40, 64), (2, 33, 1, 56, 32),
               (1, 64, 1, 64, 48), (1, 31, 2, 64, 64), (3, 97, 2, 16, 64)]


def bf16_variants():
    return [1, 2, 3, 4, 5, 6, 7, 8, 9]


@pytest.mark.parametrize("B,T,N,K,V", BF16_SHAPES)
@pytest.mark.parametrize("h0", ["zero", "uniform"])
@pytest.mark.parametrize("variant", bf16_variants())
def test_bf16_shapes(B, T, N, K, V, h0, variant):
    if not binding.variant_supports(variant, B, T, N, K, V):
        pytest.skip(f"variant {variant} does not support K={K}, V={V}")
    wl = Workload("bf16", B, T, N, K, V, h0=h0)
    check_full(wl, TOL_BF16, variant=variant, seed=B * 7 + T + K)


# Shapes off the tensor-core tile grid: K not a multiple of 16 (rows padded inside the
# kernel) and V = 48, 80, 96, 112 (readout slots padded to a power of two).
RAGGED_SHAPES = [(1, 70, 2, 1, 16), (2, 65, 1, 8, 48), (1, 130, 2, 24, 64), (1, 33, 1, 40, 80),
                 (2, 40, 1, 100, 96), (1, 70, 3, 56, 112), (1, 97, 1, 128, 112),
                 (1, 64, 1, 17, 16), (2, 33, 2, 1, 128), (1, 66, 2, 7, 32), (1, 129, 2, 127, 48),
                 (2, 20, 3, 64, 96), (1, 1, 1, 3, 80)]


@pytest.mark.parametrize("B,T,N,K,V", RAGGED_SHAPES)
@pytest.mark.parametrize("h0", ["zero", "uniform"])
def test_bf16_ragged_shapes(B, T, N, K, V, h0):
    assert binding.pick_variant(B, T, N, K, V) > 0
    wl = Workload("bf16r", B, T, N, K, V, h0=h0)
    check_full(wl, TOL_BF16, seed=B * 5 + T + K)


@pytest.mark.parametrize("B,T,N,K,V", [(2, 50, 3, 24, 48), (1, 40, 4, 1, 32)])
def test_bf16_ragged_shared_qk(B, T, N, K, V):
    wl = Workload("bf16rs", B, T, N, K, V, h0="uniform", shared_qk=True)
    check_full(wl, TOL_BF16, seed=11)


def test_bf16_small_workload_in_full():
    """B=4, T=2048, N=8, K=V=64, every output against the oracle."""
    ey, eh = check_full(WORKLOADS["b4_t2048_n8_k64_v64"], TOL_BF16)
    print(f"b4_t2048_n8_k64_v64: y err {ey:.3e}, H_T err {eh:.3e}")


SAMPLED = {
    "b8_t16384_n16_k64_v64": [(0, 0), (3, 7), (7, 15), (5, 2)],
    "b1_t65536_n16_k64_v128": [(0, 0), (0, 9), (0, 15)],
    "b16_t8192_n32_k128_v128": [(0, 0), (6, 13), (15, 31), (9, 2)],
}


@pytest.mark.slow
@pytest.mark.parametrize("name", list(SAMPLED))
def test_full_size_sampled_pairs(name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, DEV, 0)
    y, HT = run_gpu(inp)
    assert torch.isfinite(y).all() and torch.isfinite(HT).all()
    assert float(HT.abs().max()) <= 1.0 + 1e-6 or wl.h0 != "zero"
    for (b, n) in SAMPLED[name]:
        yo, HTo = m2rnn_forward_inputs(slice_pair(inp, b, n))
        ey = max_err(y[b:b + 1, :, n:n + 1], yo)
        eh = max_err(HT[b:b + 1, n:n + 1], HTo)
        print(f"{name} pair ({b},{n}): y err {ey:.3e}, H_T err {eh:.3e}")
        assert ey <= TOL_BF16 and eh <= TOL_BF16


# ---------------------------------------------------------------- invariants on the GPU
def bf16_inputs(B=2, T=150, N=2, K=64, V=64, h0="uniform", seed=3):
    return make_inputs(Workload("inv", B, T, N, K, V, h0=h0), DEV, seed)


def sub_t(inp, lo, hi):
    out = dict(inp)
    for key in ("q", "k", "v", "a"):
        out[key] = inp[key][:, lo:hi].contiguous()
    return out


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_chunked_equals_full_bitwise(dtype):
    wl = Workload("inv", 2, 150, 2, 32, 32, dtype=dtype, h0="uniform", rescale_w=dtype == "bf16")
    inp = make_inputs(wl, DEV, 4)
    y, HT = run_gpu(inp)
    first = sub_t(inp, 0, 70)
    y1, H1 = run_gpu(first)
    second = sub_t(inp, 70, 150)
    second["H0"] = H1
    y2, H2 = run_gpu(second)
    assert torch.equal(torch.cat([y1, y2], 1), y) and torch.equal(H2, HT)


def test_prefix_causality_bitwise():
    inp = bf16_inputs()
    y, _ = run_gpu(inp)
    pert = dict(inp)
    for key in ("q", "k", "v", "a"):
        x = inp[key].clone()
        x[:, 100:] = x[:, 100:] * -1.5 + 0.25
        pert[key] = x
    y2, _ = run_gpu(pert)
    assert torch.equal(y[:, :100], y2[:, :100]) and not torch.equal(y[:, 100:], y2[:, 100:])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_hold_alpha_zero_keeps_state_bitwise(dtype):
    wl = Workload("hold", 2, 40, 2, 16, 32, dtype=dtype, h0="uniform")
    inp = make_inputs(wl, DEV, 5)
    inp["alpha"] = torch.zeros_like(inp["alpha"])
    y, HT = run_gpu(inp)
    assert torch.equal(HT, inp["H0"])
    ref = (torch.einsum("bnkv,btnk->btnv", inp["H0"].double(), inp["q"].double())
           + inp["w_r"].double()[None, None] * inp["v"].double())
    tol = TOL_F32 if dtype == "f32" else 1e-5
    assert float((y.double() - ref).abs().max()) <= tol


def test_bounded_state_with_zero_h0():
    inp = bf16_inputs(h0="zero", T=300)
    inp["v"] = (inp["v"].float() * 8).to(torch.bfloat16)
    _, HT = run_gpu(inp)
    assert float(HT.abs().max()) <= 1.0


@pytest.mark.parametrize("K,V", [(16, 32), (1, 32), (1, 48)])
def test_theorem1_vector_rnn_on_gpu(K, V):
    """f -> 0, w_r = 0, q = k = e_1, H_0 = 0: y_t is the tanh RNN h_t = tanh(W^T h_{t-1} + v_t).
    K = 1 is the theorem's own case: the matrix state is a single row."""
    B, T, N = 2, 40, 2
    inp = bf16_inputs(B, T, N, K, V, h0="zero")
    e1 = torch.zeros(K, device=DEV)
    e1[0] = 1
    inp["q"] = e1.expand(B, T, N, K).to(torch.bfloat16).contiguous()
    inp["k"] = inp["q"].clone()
    inp["w_r"] = torch.zeros_like(inp["w_r"])
    inp["alpha"] = torch.full_like(inp["alpha"], 100.0)
    inp["beta"] = torch.full_like(inp["beta"], 6.0)
    inp["a"] = inp["a"].abs()
    y, HT = run_gpu(inp)
    assert torch.all(HT[:, :, 1:] == 0)
    for n in range(N):
        rnn = torch.nn.RNN(V, V, nonlinearity="tanh", bias=False, batch_first=True,
                           dtype=torch.float64)
        with torch.no_grad():
            rnn.weight_ih_l0.copy_(torch.eye(V, dtype=torch.float64))
            rnn.weight_hh_l0.copy_(inp["W"][n].double().cpu().T)
            out, _ = rnn(inp["v"][:, :, n].double().cpu())
        assert float((y[:, :, n].double().cpu() - out).abs().max()) <= TOL_BF16


# ---------------------------------------------------------------- edge cases
def test_T_zero_copies_initial_state():
    inp = bf16_inputs(T=0)
    HT = torch.empty_like(inp["H0"])
    y = torch.empty((2, 0, 2, 64), device=DEV)
    pkg.m2rnn_forward(inp, y=y, H_T=HT)
    torch.cuda.synchronize()
    assert torch.equal(HT, inp["H0"])
    inp["H0"] = None
    pkg.m2rnn_forward(inp, y=y, H_T=HT)
    torch.cuda.synchronize()
    assert torch.all(HT == 0)


def test_in_place_state_and_no_final_state():
    inp = bf16_inputs(T=90)
    y_ref, HT_ref = run_gpu(inp)
    state = inp["H0"].clone()
    inp2 = dict(inp)
    inp2["H0"] = state
    y = torch.empty_like(y_ref)
    pkg.m2rnn_forward(inp2, y=y, H_T=state)          # H0 == H_T
    assert pkg.stream_status() == binding.OK
    assert torch.equal(state, HT_ref) and torch.equal(y, y_ref)
    y3, _ = run_gpu(inp, H_T=False)                    # H_T = NULL
    assert torch.equal(y3, y_ref)


@pytest.mark.parametrize("K,V", [(129, 64), (64, 40)])
def test_unsupported_and_invalid_from_binding(K, V):
    inp = bf16_inputs(K=K, V=V, T=5)
    with pytest.raises(binding.M2RNNError) as e:
        pkg.m2rnn_forward(inp)
    assert e.value.status == binding.ERR_UNSUPPORTED


@pytest.mark.parametrize("variant,K,V", [(1, 64, 64), (2, 64, 64), (3, 128, 128), (4, 64, 128),
                                         (5, 64, 64), (6, 64, 64), (7, 128, 128), (8, 64, 128),
                                         (9, 64, 128)])
def test_forced_wait_timeout_is_reported_and_context_survives(variant, K, V):
    inp = bf16_inputs(T=70, K=K, V=V)
    y = torch.empty((2, 70, 2, V), device=DEV)
    HT = torch.empty_like(inp["H0"])
    pkg.m2rnn_forward(inp, y=y, H_T=HT, variant=variant | (1 << 8))
    assert pkg.stream_status() == binding.ERR_TIMEOUT
    assert pkg.stream_status() == binding.OK          # the word is cleared by the read
    y2, HT2 = run_gpu(inp)                            # the context is still usable
    yo, HTo = m2rnn_forward_inputs(all_f64(inp))
    assert max_err(y2, yo) <= TOL_BF16


# ---------------------------------------------------------------- balanced K = V = 128 forward
def balanced_cut_pairs(pairs, T):
    """Pairs the balanced schedule splits between two blocks (two blocks per SM)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    workers = min(pairs, 2 * sms)
    cut = []
    for w in range(workers):
        _, e = binding.balanced_stretch(pairs, T, workers, w)
        if e % T:
            cut.append(e // T)
    return cut


@pytest.mark.parametrize("B,T,N", [(3, 300, 120), (2, 100, 200), (1, 1000, 320), (2, 260, 160)])
def test_balanced_equals_one_block_per_pair_bitwise(B, T, N):
    """More pairs than resident blocks: the balanced schedule (pairs cut between blocks, the
    state handed over through y) gives the bits of one block per pair, and the cut pairs
    match the oracle."""
    wl = Workload("bal", B, T, N, 128, 128, h0="uniform")
    inp = make_inputs(wl, DEV, 21)
    y3, H3 = run_gpu(inp, variant=3)
    y7, H7 = run_gpu(inp, variant=7)
    assert torch.equal(y7, y3) and torch.equal(H7, H3)
    cut = balanced_cut_pairs(B * N, T)
    if T >= 2 * 129:
        assert cut, "expected cut pairs"
    for p in cut[:3] + cut[-1:]:
        b, n = divmod(p, N)
        yo, HTo = m2rnn_forward_inputs(slice_pair(inp, b, n))
        assert max_err(y7[b:b + 1, :, n:n + 1], yo) <= TOL_BF16
        assert max_err(H7[b:b + 1, n:n + 1], HTo) <= TOL_BF16


def test_balanced_in_place_state_no_final_state_and_shared_qk():
    wl = Workload("bal", 2, 300, 170, 128, 128, h0="uniform")
    inp = make_inputs(wl, DEV, 22)
    y_ref, HT_ref = run_gpu(inp, variant=3)
    state = inp["H0"].clone()
    inp2 = dict(inp)
    inp2["H0"] = state
    y = torch.empty_like(y_ref)
    pkg.m2rnn_forward(inp2, y=y, H_T=state, variant=7)       # H0 == H_T
    assert pkg.stream_status() == binding.OK
    assert torch.equal(state, HT_ref) and torch.equal(y, y_ref)
    y3, _ = run_gpu(inp, variant=7, H_T=False)                # H_T = NULL
    assert torch.equal(y3, y_ref)
    wls = Workload("bals", 2, 300, 170, 128, 128, h0="zero", shared_qk=True)
    inps = make_inputs(wls, DEV, 23)
    ya, Ha = run_gpu(inps, variant=3)
    yb, Hb = run_gpu(inps, variant=7)
    assert torch.equal(ya, yb) and torch.equal(Ha, Hb)


def test_balanced_forced_timeout_with_cut_pairs():
    wl = Workload("bal", 2, 300, 160, 128, 128, h0="uniform")
    inp = make_inputs(wl, DEV, 24)
    y = torch.empty((2, 300, 160, 128), device=DEV)
    HT = torch.empty_like(inp["H0"])
    pkg.m2rnn_forward(inp, y=y, H_T=HT, variant=7 | (1 << 8))
    assert pkg.stream_status() == binding.ERR_TIMEOUT
    assert pkg.stream_status() == binding.OK
    y3, H3 = run_gpu(inp, variant=3)
    y7, H7 = run_gpu(inp, variant=7)
    assert torch.equal(y7, y3) and torch.equal(H7, H3)


@pytest.mark.parametrize("variant,N,K,V", [(3, 160, 128, 128), (7, 160, 128, 128),
                                           (8, 3, 64, 128), (9, 3, 64, 128)])
def test_tcgen05_forward_cuda_graph_replay(variant, N, K, V):
    """The forward captured in a CUDA graph and replayed: every replay gives the eager bits,
    also for the balanced schedule, whose handoff tags carry the epoch of the captured launch
    (each replay's taking block overwrites them with y before the next), and for the 8-SM-per-
    pair kernels (whose launcher queries the occupancy calculator; the two-cluster form also
    zeroes y before its clusters add into it)."""
    wl = Workload("gr", 2, 300, N, K, V, h0="uniform")
    inp = make_inputs(wl, DEV, 31)
    y_ref, HT_ref = run_gpu(inp, variant=variant)
    y = torch.full_like(y_ref, float("nan"))
    HT = torch.full_like(HT_ref, float("nan"))
    pkg.m2rnn_forward(inp, y=y, H_T=HT, variant=variant)    # first call outside capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            pkg.m2rnn_forward(inp, y=y, H_T=HT, variant=variant, stream=s)
    for _ in range(3):
        y.fill_(float("nan"))
        HT.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pkg.stream_status() == binding.OK
        assert torch.equal(y, y_ref) and torch.equal(HT, HT_ref)


@pytest.mark.parametrize("variant", [8, 9])
@pytest.mark.parametrize("B,T,N", [(1, 96, 2), (2, 33, 1), (1, 257, 3)])
def test_cluster8_in_place_state_no_final_state_and_chunks(B, T, N, variant):
    """The eight-SMs-per-pair kernels (K = 64, V = 128; one 8-CTA cluster, or two 4-CTA
    clusters adding into y): in-place state (H0 == H_T), no final state, and a sequence run as
    two calls (the state carried through H_T) give the bits of one call; chunk-boundary
    lengths (32-step chunks) included.  The two forms differ only in the order of the readout
    sums over rows."""
    inp = bf16_inputs(B=B, T=T, N=N, K=64, V=128)
    y_ref, HT_ref = run_gpu(inp, variant=variant)
    state = inp["H0"].clone()
    inp2 = dict(inp)
    inp2["H0"] = state
    y = torch.empty_like(y_ref)
    pkg.m2rnn_forward(inp2, y=y, H_T=state, variant=variant)       # H0 == H_T
    assert pkg.stream_status() == binding.OK
    assert torch.equal(state, HT_ref) and torch.equal(y, y_ref)
    y3, _ = run_gpu(inp, variant=variant, H_T=False)               # H_T = NULL
    assert torch.equal(y3, y_ref)
    cut = 64 if T > 64 else T // 2
    ya, Ha = run_gpu(sub_t(inp, 0, cut), variant=variant)
    rest = sub_t(inp, cut, T)
    rest["H0"] = Ha
    yb, Hb = run_gpu(rest, variant=variant)
    assert torch.equal(torch.cat([ya, yb], dim=1), y_ref) and torch.equal(Hb, HT_ref)
    if variant == 9:   # the same state arithmetic as one 8-CTA cluster per pair
        y8, H8 = run_gpu(inp, variant=8)
        assert torch.equal(H8, HT_ref)
        assert float((y8 - y_ref).abs().max()) <= 1e-5
