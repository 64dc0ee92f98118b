"""Decode step (T = 1, state in / state out) on the GPU.

The decode kernel performs exactly one step of the warp-MMA forward kernels' arithmetic
(the pipelined kernel, variant 2, where it applies, else the row-warp kernel, variant 1),
so:
  * one call equals that forward over a single token, bit for bit;
  * T calls with the state updated in place equal a T-step forward, bit for bit
    (every y_t and the final state);
and it matches the fp64 oracle within the bf16 path's 3e-2.  A CUDA graph of
several decode steps replays to the same bits as the eager calls.
"""
import numpy as np
import pytest
import torch

import __graft_entry__
import matrix_state_nonlinear_gb300 as pkg
from matrix_state_nonlinear_gb300 import m2rnn as binding
from matrix_state_nonlinear_gb300.inputs import Workload, all_f64, make_inputs
from oracle import m2rnn_forward_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    __graft_entry__.build()
    pkg.load_library()


def twin(inp, K, V):
    """The forward pass whose arithmetic the decode kernel reproduces step by step."""
    variant = 2 if binding.variant_supports(2, 1, 1, 1, K, V) else 1
    return pkg.m2rnn_forward(inp, variant=variant)


def step_args(inp, t):
    return (inp["q"][:, t].contiguous(), inp["k"][:, t].contiguous(), inp["v"][:, t].contiguous(),
            inp["a"][:, t].contiguous(), inp["alpha"], inp["beta"], inp["W"], inp["w_r"])


@pytest.mark.parametrize("shape,shared", [((2, 37, 3, 64, 64), False), ((3, 20, 2, 32, 16), False),
                                          ((2, 9, 4, 48, 32), True), ((1, 70, 2, 16, 64), False),
                                          ((96, 3, 8, 64, 64), False), ((40, 2, 16, 32, 16), True),
                                          ((70, 2, 9, 48, 32), False),
                                          # ragged K and V (row-warp forward)
                                          ((2, 9, 3, 24, 48), False), ((3, 5, 2, 1, 16), True),
                                          ((2, 6, 2, 100, 96), False), ((2, 4, 2, 40, 80), False),
                                          # >= 2048 pairs at K = V = 64: the persistent kernel
                                          ((160, 2, 16, 64, 64), False), ((130, 3, 16, 64, 64), True)])
def test_decode_steps_reproduce_the_forward_bitwise(shape, shared):
    B, T, N, K, V = shape
    inp = make_inputs(Workload("dec", B, T, N, K, V, h0="uniform", shared_qk=shared), DEV, 5)
    y_ref, H_ref = twin(inp, K, V)
    H = inp["H0"].clone()
    for t in range(T):
        y, _ = pkg.m2rnn_decode_step(*step_args(inp, t), H)   # in place
        assert torch.equal(y, y_ref[:, t]), t
    assert pkg.stream_status() == binding.OK
    assert torch.equal(H, H_ref)


@pytest.mark.parametrize("shape", [(2, 5, 3, 128, 64), (4, 3, 2, 112, 16), (2, 6, 3, 64, 128),
                                   (2, 4, 2, 128, 128), (1, 3, 1, 32, 128)])
def test_decode_large_K_matches_oracle(shape):
    B, T, N, K, V = shape
    inp = make_inputs(Workload("decK", B, T, N, K, V, h0="uniform"), DEV, 6)
    H = inp["H0"].clone()
    ys = []
    for t in range(T):
        y, _ = pkg.m2rnn_decode_step(*step_args(inp, t), H)
        ys.append(y.clone())
    yo, Ho = m2rnn_forward_inputs(all_f64(inp))
    err_y = float(np.abs(torch.stack(ys, 1).double().cpu().numpy() - yo).max())
    err_h = float(np.abs(H.double().cpu().numpy() - Ho).max())
    assert err_y <= 3e-2 and err_h <= 3e-2, (err_y, err_h)


@pytest.mark.parametrize("B, N", [(3, 2), (256, 8)])   # 512 and 2048 pairs
def test_decode_zero_state_and_separate_output(B, N):
    inp = make_inputs(Workload("dec0", B, 1, N, 64, 64, h0="zero"), DEV, 7)
    y_ref, H_ref = twin(inp, 64, 64)
    H_out = torch.full((B, N, 64, 64), float("nan"), device=DEV)
    y, _ = pkg.m2rnn_decode_step(*step_args(inp, 0), None, H_out=H_out)
    assert pkg.stream_status() == binding.OK
    assert torch.equal(y, y_ref[:, 0]) and torch.equal(H_out, H_ref)


@pytest.mark.parametrize("B, N", [(4, 4), (128, 16)])   # 16 pairs; 2048 pairs (persistent kernel)
def test_decode_cuda_graph_replay(B, N):
    T, K, V = 8, 64, 64
    inp = make_inputs(Workload("decg", B, T, N, K, V, h0="uniform"), DEV, 8)
    steps = [step_args(inp, t) for t in range(T)]
    H_eager = inp["H0"].clone()
    ys_eager = [pkg.m2rnn_decode_step(*steps[t], H_eager)[0].clone() for t in range(T)]
    H = inp["H0"].clone()
    ys = [torch.empty((B, N, V), device=DEV) for _ in range(T)]
    pkg.m2rnn_decode_step(*steps[0], H.clone(), y=ys[0])       # first call outside capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            for t in range(T):
                pkg.m2rnn_decode_step(*steps[t], H, y=ys[t], stream=s)
    H.copy_(inp["H0"])
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(H, H_eager)
    for t in range(T):
        assert torch.equal(ys[t], ys_eager[t]), t


@pytest.mark.parametrize("B, N", [(4, 4), (160, 16)])   # 16 pairs; 2560 pairs
def test_decode_kernels_agree_bitwise(B, N):
    """The per-pair kernel and the persistent kernel (forced at any pair count) give the
    same bits."""
    inp = make_inputs(Workload("decv", B, 1, N, 64, 64, h0="uniform"), DEV, 9)
    outs = []
    for variant in (1, 2):
        H = torch.empty_like(inp["H0"])
        y, _ = pkg.m2rnn_decode_step(*step_args(inp, 0), inp["H0"], H_out=H, variant=variant)
        assert pkg.stream_status() == binding.OK
        outs.append((y, H))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_persistent_decode_forced_timeout_is_reported_and_context_survives():
    """The persistent kernel's bounded wait gives up on a barrier nothing arrives at: the
    status word reports the timeout, the read clears it, and the next decode is still
    bit-identical to the forward."""
    B, N, T = 128, 16, 2                                  # 2048 pairs
    inp = make_inputs(Workload("decto", B, T, N, 64, 64, h0="uniform"), DEV, 10)
    H = inp["H0"].clone()
    y = torch.empty((B, N, 64), device=DEV)
    pkg.m2rnn_decode_step(*step_args(inp, 0), H, y=y, variant=2 | (1 << 8))
    assert pkg.stream_status() == binding.ERR_TIMEOUT
    assert pkg.stream_status() == binding.OK
    y_ref, H_ref = twin(inp, 64, 64)
    H = inp["H0"].clone()
    for t in range(T):
        y, _ = pkg.m2rnn_decode_step(*step_args(inp, t), H, variant=2)
        assert torch.equal(y, y_ref[:, t]), t
    assert pkg.stream_status() == binding.OK
    assert torch.equal(H, H_ref)
