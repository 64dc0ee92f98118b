"""Training support on the GPU: the state-keeping forward and the backward pass
against the fp64 oracle (the notes' Sec. 2.6-2.7), through the C ABI.

Tolerances (max-abs error per gradient tensor, scaled by max(1, max |oracle|)):
  * fp32 path: 1e-4.  Every step is fp32 with accurate tanh/exp; the reverse scan
    adds one rounding per operation along T steps, far below 1e-4 at these sizes.
  * bf16 path: 3e-2.  The kept states come from the bf16-operand forward, whose
    states differ from the exact ones by up to its own bar (3e-2), and are kept
    rounded to bf16 (relative 2^-9); the gradients are smooth in the states, so
    they carry errors of the same relative size.
"""
import numpy as np
import pytest
import torch

import __graft_entry__
import matrix_state_nonlinear_gb300 as pkg
from matrix_state_nonlinear_gb300 import m2rnn as binding
from matrix_state_nonlinear_gb300.inputs import Workload, all_f64, make_inputs
from oracle import m2rnn_backward_inputs, m2rnn_forward_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = {"f32": 1e-4, "bf16": 3e-2}
GRADS = ["dq", "dk", "dv", "da", "dalpha", "dbeta", "dW", "dw_r", "dH0"]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    __graft_entry__.build()
    pkg.load_library()


def upstream(B, T, N, K, V, seed, with_dHT=True):
    g = torch.Generator(device="cpu").manual_seed(seed)
    dy = torch.randn((B, T, N, V), generator=g).to(DEV)
    dHT = torch.randn((B, N, K, V), generator=g).to(DEV) if with_dHT else None
    return dy, dHT


def rel_err(got, want):
    got = got.double().cpu().numpy() if torch.is_tensor(got) else np.asarray(got)
    want = np.asarray(want, np.float64)
    return float(np.abs(got - want).max()) / max(1.0, float(np.abs(want).max())) if want.size else 0.0


def run_case(dtype, B, T, N, K, V, h0="uniform", shared=False, with_dHT=True, seed=0, variant=0):
    wl = Workload("bwd", B, T, N, K, V, dtype=dtype, h0=h0, shared_qk=shared,
                  rescale_w=dtype == "bf16")
    inp = make_inputs(wl, DEV, seed)
    y, HT, Hs = pkg.m2rnn_forward_train(inp)
    dy, dHT = upstream(B, T, N, K, V, seed + 1, with_dHT)
    g = pkg.m2rnn_backward(inp, Hs, dy, dHT, variant=variant)
    assert pkg.stream_status() == binding.OK
    ref = m2rnn_backward_inputs(all_f64(inp), dy.double().cpu().numpy(),
                                None if dHT is None else dHT.double().cpu().numpy())
    errs = {n: rel_err(g[n], ref[n]) for n in GRADS}
    return inp, (y, HT, Hs), g, errs


F32_SHAPES = [(1, 1, 1, 1, 1), (2, 5, 3, 8, 8), (1, 64, 2, 8, 8), (1, 17, 2, 24, 40),
              (2, 33, 1, 16, 128), (1, 9, 1, 128, 128), (3, 2, 2, 5, 7)]


@pytest.mark.parametrize("shape", F32_SHAPES)
@pytest.mark.parametrize("h0", ["zero", "uniform"])
def test_backward_f32_matches_oracle(shape, h0):
    _, _, _, errs = run_case("f32", *shape, h0=h0)
    assert max(errs.values()) <= TOL["f32"], errs


@pytest.mark.parametrize("shape", [(2, 7, 3, 8, 16), (1, 20, 4, 16, 8)])
def test_backward_f32_shared_qk(shape):
    _, _, g, errs = run_case("f32", *shape, shared=True)
    assert g["dq"].shape[2] == 1
    assert max(errs.values()) <= TOL["f32"], errs


def test_backward_without_dHT_and_without_dH0():
    wl = Workload("bwd", 2, 11, 2, 8, 8, dtype="f32", rescale_w=False, h0="uniform")
    inp = make_inputs(wl, DEV, 4)
    _, _, Hs = pkg.m2rnn_forward_train(inp)
    dy, _ = upstream(2, 11, 2, 8, 8, 5, False)
    lib = binding.load_library()
    g = pkg.m2rnn_backward(inp, Hs, dy)
    ref = m2rnn_backward_inputs(all_f64(inp), dy.double().cpu().numpy())
    assert max(rel_err(g[n], ref[n]) for n in GRADS) <= TOL["f32"]
    # dH0 == NULL: everything else is unchanged
    grads = {n: torch.full_like(g[n], float("nan")) for n in GRADS if n != "dH0"}
    out = {n: grads[n] for n in grads}
    ws = torch.empty(binding.backward_workspace_bytes(2, 11, 2, 2, 8, 8), dtype=torch.uint8,
                     device=DEV)
    args = [inp[x] for x in ("q", "k", "v", "a", "alpha", "beta", "W", "w_r", "H0")]
    st = lib.m2rnn_backward_f32(*[t.data_ptr() for t in args], Hs.data_ptr(), dy.data_ptr(), None,
                                *[out[n].data_ptr() for n in GRADS if n != "dH0"], None,
                                2, 11, 2, 2, 8, 8, ws.data_ptr(), ws.numel(), None)
    assert st == binding.OK and pkg.stream_status() == binding.OK
    for n in out:
        assert torch.equal(out[n], g[n]), n


def test_forward_train_keeps_states_and_matches_plain_forward():
    # The bf16 state-keeping forward runs the pipelined kernel's arithmetic (forward variant
    # 2) for K, V <= 64 with K % 16 == 0, the tcgen05 kernel's (variant 3, or its balanced
    # form 7 above two pairs per SM) for K = V = 128, eight SMs per pair for K = 64, V = 128
    # (one 8-CTA cluster, variant 8, while all fit; else two 4-CTA clusters, variant 9; else the
    # 4-CTA kernel, 4), and the row-warp kernel's (variant 1) otherwise.
    for dtype, shape, fwd_variant in [("f32", (2, 37, 3, 8, 24), 0), ("bf16", (2, 150, 3, 64, 64), 2),
                                      ("bf16", (1, 70, 2, 32, 16), 2),
                                      ("bf16", (2, 45, 2, 64, 128), 8),   # 8-CTA cluster
                                      ("bf16", (1, 41, 16, 64, 128), 9),  # 16 pairs: 2 x 4-CTA
                                      ("bf16", (1, 33, 2, 128, 128), 3),   # tcgen05
                                      # ragged K and V off the power-of-two grid (row-warp)
                                      ("bf16", (2, 40, 2, 24, 48), 1),
                                      ("bf16", (1, 30, 1, 100, 112), 1),
                                      ("bf16", (1, 20, 3, 1, 16), 1)]:
        B, T, N, K, V = shape
        wl = Workload("tr", B, T, N, K, V, dtype=dtype, h0="uniform", rescale_w=dtype == "bf16")
        inp = make_inputs(wl, DEV, 7)
        y, HT, Hs = pkg.m2rnn_forward_train(inp)
        y2, HT2 = pkg.m2rnn_forward(inp, variant=fwd_variant)
        assert torch.equal(y, y2) and torch.equal(HT, HT2)     # same arithmetic, bit for bit
        assert torch.equal(Hs[:, :, T - 1], HT.to(Hs.dtype))    # bf16: round to nearest even
        _, _, states = m2rnn_forward_inputs(all_f64(inp), return_states=True)
        err = float(np.abs(Hs.double().cpu().numpy() - np.moveaxis(states, 1, 2)).max())
        assert err <= TOL[dtype], err


def test_forward_train_balanced_keeps_states():
    """K = V = 128 with more pairs than two per SM: the state-keeping forward runs the balanced
    schedule (pairs cut between blocks, the state handed over mid-sequence); its y and H_T are
    the plain forward's bits, and the kept states of cut pairs, on both sides of the cut,
    match the oracle's."""
    B, T, N, K, V = 2, 300, 170, 128, 128
    wl = Workload("trb", B, T, N, K, V, h0="uniform")
    inp = make_inputs(wl, DEV, 12)
    y, HT, Hs = pkg.m2rnn_forward_train(inp)
    assert pkg.stream_status() == binding.OK
    y3, HT3 = pkg.m2rnn_forward(inp, variant=3)
    assert torch.equal(y, y3) and torch.equal(HT, HT3)
    assert torch.equal(Hs[:, :, T - 1], HT.to(Hs.dtype))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    workers = min(B * N, 2 * sms)
    cut = [e // T for e in (binding.balanced_stretch(B * N, T, workers, w)[1]
                            for w in range(workers)) if e % T]
    assert cut
    from matrix_state_nonlinear_gb300.inputs import slice_pair
    for p in cut[:2]:
        b, n = divmod(p, N)
        _, _, states = m2rnn_forward_inputs(slice_pair(inp, b, n), return_states=True)
        err = float(np.abs(Hs[b, n].double().cpu().numpy() - states[0, :, 0]).max())
        assert err <= TOL["bf16"], (p, err)


BF16_SHAPES = [(1, 1, 1, 16, 16), (2, 65, 3, 64, 64), (1, 130, 2, 32, 32), (2, 40, 2, 48, 16),
               (1, 1, 1, 64, 64), (1, 4, 2, 64, 64), (1, 5, 1, 64, 64), (2, 131, 2, 64, 64),
               (1, 7, 2, 64, 64), (1, 24, 2, 64, 128), (1, 12, 1, 128, 128), (1, 10, 2, 96, 128),
               # chunk edges of the 8-step backward chunks: exactly one, one plus one step,
               # exactly two, and a two-step sequence
               (1, 8, 2, 64, 64), (1, 9, 1, 64, 64), (1, 16, 2, 64, 64), (2, 2, 1, 64, 64),
               # ragged K, V of 48 / 80 (row-warp state-keeping forward, SIMT backward)
               (1, 20, 2, 24, 48), (2, 15, 1, 1, 80),
               # V = 128 on the tensor-core backward: one, two, three and four steps (the state
               # ring's start), rows padded from K = 16, 32, 48, 64, 96 to 128
               (1, 1, 1, 16, 128), (1, 2, 1, 32, 128), (2, 3, 1, 128, 128), (1, 4, 1, 64, 128),
               (2, 37, 2, 48, 128), (1, 70, 1, 128, 128)]


def bwd_variants(K, V):
    # 1: SIMT (any shape); 2: warp-MMA kernel; 3, 4: tcgen05 kernels with 4 or 8 compute
    # warps; 5: every product on tcgen05, the chain included (K = V = 64); 6: every product
    # on tcgen05 for V = 128 (K a multiple of 16, rows padded); 7: the same with the
    # recurrence's products transposed (V = 128, K <= 64)
    if (K, V) == (64, 64):
        return [1, 2, 3, 4, 5]
    if V == 128 and K % 16 == 0:
        return [1, 6, 7] if K <= 64 else [1, 6]
    return [1]


@pytest.mark.parametrize("shape", BF16_SHAPES)
@pytest.mark.parametrize("h0", ["zero", "uniform"])
def test_backward_bf16_matches_oracle(shape, h0):
    for variant in bwd_variants(shape[3], shape[4]):
        _, _, _, errs = run_case("bf16", *shape, h0=h0, variant=variant)
        assert max(errs.values()) <= TOL["bf16"], (variant, errs)


def kv_of(variant):
    return (64, 128) if variant in (6, 7) else (64, 64)


@pytest.mark.parametrize("variant", [1, 2, 3, 4, 5, 6, 7])
def test_backward_bf16_shared_qk(variant):
    _, _, g, errs = run_case("bf16", 2, 50, 4, *kv_of(variant), shared=True, variant=variant)
    assert g["dq"].shape[2] == 1
    assert max(errs.values()) <= TOL["bf16"], errs


@pytest.mark.parametrize("variant", [2, 3, 4, 5, 6, 7])
def test_backward_mma_without_dHT(variant):
    _, _, _, errs = run_case("bf16", 2, 37, 2, *kv_of(variant), with_dHT=False, variant=variant)
    assert max(errs.values()) <= TOL["bf16"], errs


@pytest.mark.parametrize("variant", [2, 3, 4, 5, 6, 7])
def test_backward_mma_close_to_simt(variant):
    """The kernels differentiate the same kept states; they differ only by rounding
    (bf16 D in the MMA products vs fp32 SIMT sums)."""
    K, V = kv_of(variant)
    wl = Workload("cmp", 2, 90, 3, K, V, h0="uniform")
    inp = make_inputs(wl, DEV, 8)
    _, _, Hs = pkg.m2rnn_forward_train(inp)
    dy, dHT = upstream(2, 90, 3, K, V, 9)
    g1 = pkg.m2rnn_backward(inp, Hs, dy, dHT, variant=1)
    g2 = pkg.m2rnn_backward(inp, Hs, dy, dHT, variant=variant)
    for n in GRADS:
        assert rel_err(g2[n], g1[n].double().cpu().numpy()) <= 1e-2, n


@pytest.mark.parametrize("variant", [2, 3, 4, 5, 6, 7])
def test_backward_mma_forced_timeout_is_reported(variant):
    K, V = kv_of(variant)
    wl = Workload("to", 2, 20, 2, K, V, h0="uniform")
    inp = make_inputs(wl, DEV, 3)
    _, _, Hs = pkg.m2rnn_forward_train(inp)
    dy, dHT = upstream(2, 20, 2, K, V, 4)
    pkg.m2rnn_backward(inp, Hs, dy, dHT, variant=variant | (1 << 8))
    assert pkg.stream_status() == binding.ERR_TIMEOUT
    assert pkg.stream_status() == binding.OK
    g = pkg.m2rnn_backward(inp, Hs, dy, dHT, variant=variant)   # the context still works
    ref = m2rnn_backward_inputs(all_f64(inp), dy.double().cpu().numpy(),
                                dHT.double().cpu().numpy())
    assert max(rel_err(g[n], ref[n]) for n in GRADS) <= TOL["bf16"]


def test_backward_is_deterministic():
    wl = Workload("det", 3, 40, 2, 16, 32, dtype="bf16", h0="uniform")
    inp = make_inputs(wl, DEV, 2)
    _, _, Hs = pkg.m2rnn_forward_train(inp)
    dy, dHT = upstream(3, 40, 2, 16, 32, 3)
    g1 = pkg.m2rnn_backward(inp, Hs, dy, dHT)
    g2 = pkg.m2rnn_backward(inp, Hs, dy, dHT)
    for n in GRADS:
        assert torch.equal(g1[n], g2[n]), n


def test_backward_empty_sequence():
    wl = Workload("e", 2, 0, 2, 8, 8, dtype="f32", h0="uniform", rescale_w=False)
    inp = make_inputs(wl, DEV, 1)
    Hs = torch.empty((2, 2, 0, 8, 8), device=DEV)      # fp32 path: float32 states
    dy = torch.empty((2, 0, 2, 8), device=DEV)
    dHT = torch.randn((2, 2, 8, 8), device=DEV)
    g = pkg.m2rnn_backward(inp, Hs, dy, dHT)
    assert pkg.stream_status() == binding.OK
    assert torch.equal(g["dH0"], dHT)
    for n in ("dW", "dw_r", "dalpha", "dbeta"):
        assert float(g[n].abs().max()) == 0.0


def abs_err(got, want):
    got = got.double().cpu().numpy() if torch.is_tensor(got) else np.asarray(got)
    want = np.asarray(want, np.float64)
    return float(np.abs(got - want).max()) if want.size else 0.0


@pytest.mark.slow
@pytest.mark.parametrize("shape,shared,variant", [
    # the training workload's length and head shape on the tensor-core backward (auto = 5)
    ((1, 16384, 4, 64, 64), False, 0),
    ((1, 16384, 4, 64, 64), True, 0),
    # V = 128 at long T on its tensor-core backwards (auto = 7 for K <= 64, else 6; both
    # forms at K = 64), per-head and shared q, k
    ((1, 4096, 2, 64, 128), False, 0),
    ((1, 4096, 2, 64, 128), False, 6),
    ((1, 1024, 3, 32, 128), True, 7),
    ((1, 2048, 2, 128, 128), True, 0),
])
def test_backward_bf16_at_training_length(shape, shared, variant):
    """Every gradient tensor against the fp64 backward oracle over the whole sequence:
    thousands of wraps of the 8-step chunk ring and of the state-history stream, so an
    error that grows along the reverse scan would show.  The bar is the bf16 path's 3e-2
    on the max-abs error scaled by max(1, max |oracle|); the unscaled max-abs error and
    the oracle's magnitude are printed beside it."""
    B, T, N, K, V = shape
    wl = Workload("bwdT", B, T, N, K, V, h0="zero", shared_qk=shared)
    inp = make_inputs(wl, DEV, 21)
    _, _, Hs = pkg.m2rnn_forward_train(inp)
    dy, dHT = upstream(B, T, N, K, V, 22)
    g = pkg.m2rnn_backward(inp, Hs, dy, dHT, variant=variant)
    assert pkg.stream_status() == binding.OK
    ref = m2rnn_backward_inputs(all_f64(inp), dy.double().cpu().numpy(),
                                dHT.double().cpu().numpy())
    worst = 0.0
    for n in GRADS:
        scaled, unscaled = rel_err(g[n], ref[n]), abs_err(g[n], ref[n])
        mag = float(np.abs(np.asarray(ref[n])).max())
        print(f"{shape} shared={shared} {n}: scaled {scaled:.3e}  max-abs {unscaled:.3e}  "
              f"max|oracle| {mag:.3e}")
        worst = max(worst, scaled)
    assert worst <= TOL["bf16"]
