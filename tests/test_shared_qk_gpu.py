"""Multi-value sharing on the GPU (one q, k set for all heads; the M²RNN notes' Sec. 2.4).

Every kernel variant's shared-q/k result must equal, bitwise, its own result with
the shared vectors tiled over the heads (the kernels do the same arithmetic on the
same values), and match the fp64 oracle within the path's tolerance.
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


def run(inp, variant):
    B, T, _, K = inp["q"].shape
    N, V = inp["v"].shape[2], inp["v"].shape[3]
    y = torch.full((B, T, N, V), float("nan"), device=DEV)
    HT = torch.full((B, N, K, V), float("nan"), device=DEV)
    pkg.m2rnn_forward(inp, y=y, H_T=HT, variant=variant)
    assert pkg.stream_status() == binding.OK
    return y, HT


CASES = [("f32", 0, (2, 33, 3, 8, 8)), ("bf16", 1, (2, 70, 3, 32, 32)), ("bf16", 1, (1, 40, 2, 64, 128)),
         ("bf16", 2, (2, 97, 3, 64, 64)), ("bf16", 2, (1, 66, 4, 16, 32)), ("bf16", 3, (2, 40, 3, 128, 128)),
         ("bf16", 4, (1, 150, 3, 64, 128)), ("bf16", 5, (2, 97, 3, 64, 64)),
         ("bf16", 5, (1, 66, 4, 32, 48)), ("bf16", 6, (2, 97, 3, 64, 64)),
         ("bf16", 6, (1, 70, 2, 64, 16)), ("bf16", 8, (1, 150, 3, 64, 128)),
         ("bf16", 9, (1, 150, 3, 64, 128))]


@pytest.mark.parametrize("dtype,variant,shape", CASES)
def test_shared_qk_matches_tiled_and_oracle(dtype, variant, shape):
    B, T, N, K, V = shape
    wl = Workload("sqk", B, T, N, K, V, dtype=dtype, h0="uniform", shared_qk=True,
                  rescale_w=dtype == "bf16")
    inp = make_inputs(wl, DEV, 9)
    assert inp["q"].shape == (B, T, 1, K)
    y, HT = run(inp, variant)
    tiled = dict(inp)
    tiled["q"] = inp["q"].expand(B, T, N, K).contiguous()
    tiled["k"] = inp["k"].expand(B, T, N, K).contiguous()
    y2, HT2 = run(tiled, variant)
    assert torch.equal(y, y2) and torch.equal(HT, HT2)
    yo, HTo = m2rnn_forward_inputs(all_f64(inp))
    tol = 1e-4 if dtype == "f32" else 3e-2
    ey = float(np.abs(y.double().cpu().numpy() - yo).max())
    eh = float(np.abs(HT.double().cpu().numpy() - HTo).max())
    assert ey <= tol and eh <= tol, (ey, eh)
