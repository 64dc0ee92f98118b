"""m2rnn_backward_bf16_noalloc: the bf16 backward with the library's fixed scratch.

Named to sort last, so that in a full run it executes after every other test (and
it also passes alone).  The GPU tests make two calls in a row on the same scratch
and compare both with the workspace entry point (bit for bit) and with the oracle.
"""
import numpy as np
import pytest
import torch

import __graft_entry__
import matrix_state_nonlinear_gb300 as pkg
from matrix_state_nonlinear_gb300 import m2rnn as binding
from matrix_state_nonlinear_gb300.inputs import Workload, all_f64, make_inputs
from oracle import m2rnn_backward_inputs

GRADS = ["dq", "dk", "dv", "da", "dalpha", "dbeta", "dW", "dw_r", "dH0"]
SCRATCH_BYTES = 16 << 20


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return binding.load_library()


def test_oversized_request_is_refused_before_the_device(lib):
    # B=8, T=16384, N=16, K=V=64 with shared q, k needs about 1 GiB of workspace.
    assert binding.backward_workspace_bytes(8, 16384, 16, 1, 64, 64) > SCRATCH_BYTES
    p = [(1 << 20) + 256 * i for i in range(21)]
    st = lib.m2rnn_backward_bf16_noalloc(*p, 8, 16384, 16, 1, 64, 64, None)
    assert st == binding.ERR_UNSUPPORTED
    st = lib.m2rnn_backward_bf16_noalloc(*p, 1, 4, 2, 3, 16, 16, None)   # Nqk not 1 or N
    assert st == binding.ERR_INVALID_ARG


@pytest.mark.gpu
def test_two_calls_in_a_row_match_the_workspace_path(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = "cuda:0"
    cases = [Workload("na1", 2, 70, 3, 64, 64, h0="uniform"),
             Workload("na2", 1, 33, 2, 32, 16, h0="zero", shared_qk=True)]
    for i, wl in enumerate(cases):
        inp = make_inputs(wl, dev, 20 + i)
        _, _, Hs = pkg.m2rnn_forward_train(inp)
        gen = torch.Generator(device="cpu").manual_seed(30 + i)
        dy = torch.randn((wl.B, wl.T, wl.N, wl.V), generator=gen).to(dev)
        dHT = torch.randn((wl.B, wl.N, wl.K, wl.V), generator=gen).to(dev)
        ref_ws = pkg.m2rnn_backward(inp, Hs, dy, dHT)
        first = binding.m2rnn_backward_noalloc(inp, Hs, dy, dHT)
        second = binding.m2rnn_backward_noalloc(inp, Hs, dy, dHT)
        assert pkg.stream_status() == binding.OK
        for n in GRADS:
            assert torch.equal(first[n], ref_ws[n]), n
            assert torch.equal(second[n], ref_ws[n]), n
        ref = m2rnn_backward_inputs(all_f64(inp), dy.double().cpu().numpy(),
                                    dHT.double().cpu().numpy())
        for n in GRADS:
            want = ref[n]
            err = float(np.abs(second[n].double().cpu().numpy() - want).max())
            assert err <= 3e-2 * max(1.0, float(np.abs(want).max())), (n, err)
