"""The block's prologue (causal Conv1D k=4 + SiLU) and epilogue (gate + RMSNorm) on the
GPU against the fp64 oracle (the M²RNN notes' Sec. 2.3), and the three stages chained
around the recurrence.

Tolerances: both kernels compute in fp32 and round once to bf16, so each output is
within half a bf16 ulp of the exact value plus fp32 rounding: |gpu - oracle| <=
2^-8 |oracle| + 1e-5.  The chained block is checked stage by stage: the readout from
the GPU's convolved q, k, v against the oracle's (conv outputs rounded to bf16, nearest
even, like the GPU's) at the recurrence's bf16 bar (3e-2), then the epilogue on that
readout at the rounding bound.
"""
import numpy as np
import pytest
import torch

import __graft_entry__
import matrix_state_nonlinear_gb300 as pkg
from matrix_state_nonlinear_gb300 import m2rnn as binding
from matrix_state_nonlinear_gb300.inputs import Workload, all_f64, make_inputs
from oracle import conv_silu, gate_rmsnorm, m2rnn_forward_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    __graft_entry__.build()
    pkg.load_library()


def close_bf16(got, want):
    got = got.double().cpu().numpy()
    return float(np.max(np.abs(got - want) - (2.0 ** -8 * np.abs(want) + 1e-5)))


def rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16).to(DEV)


@pytest.mark.parametrize("shape", [(1, 1, 8), (2, 3, 16), (2, 70, 24), (3, 200, 64), (1, 129, 1024)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_conv_silu_matches_oracle(shape, with_bias):
    B, T, C = shape
    x = rand_bf16(shape, 1, 1.5)
    w = (torch.randn((C, 4), generator=torch.Generator().manual_seed(2)) * 0.6).to(DEV)
    bias = (torch.randn(C, generator=torch.Generator().manual_seed(3)) * 0.3).to(DEV) if with_bias else None
    out = pkg.conv_silu(x, w, bias)
    assert pkg.stream_status() == binding.OK
    ref = conv_silu(x.double().cpu().numpy(), w.double().cpu().numpy(),
                    None if bias is None else bias.double().cpu().numpy())
    assert close_bf16(out, ref) <= 0.0


@pytest.mark.parametrize("rows,D", [(1, 8), (5, 64), (7, 1024), (3, 1000), (33, 2048)])
@pytest.mark.parametrize("eps", [0.0, 1e-6])
def test_gate_rmsnorm_matches_oracle(rows, D, eps):
    g = torch.Generator().manual_seed(rows + D)
    y = torch.randn((rows, D), generator=g).to(DEV)
    gp = rand_bf16((rows, D), rows * 7 + D)
    wn = (1.0 + 0.1 * torch.randn(D, generator=g)).to(DEV)
    out = pkg.gate_rmsnorm(y, gp, wn, eps)
    assert pkg.stream_status() == binding.OK
    ref = gate_rmsnorm(y.double().cpu().numpy(), gp.double().cpu().numpy(),
                       wn.double().cpu().numpy(), eps)
    assert close_bf16(out, ref) <= 0.0


def test_block_chain_matches_oracle():
    B, T, N, K, V = 2, 150, 4, 64, 64
    wl = Workload("blk", B, T, N, K, V, h0="zero")
    inp = make_inputs(wl, DEV, 3)
    pre = {n: rand_bf16((B, T, N * (V if n == "v" else K)), 10 + i, 1.0)
           for i, n in enumerate(["q", "k", "v"])}
    cw = {n: (torch.randn((pre[n].shape[2], 4), generator=torch.Generator().manual_seed(20 + i))
              * 0.5).to(DEV) for i, n in enumerate(["q", "k", "v"])}
    gpre = rand_bf16((B, T, N * V), 30)
    wn = (1.0 + 0.1 * torch.randn(N * V, generator=torch.Generator().manual_seed(31))).to(DEV)
    # GPU: prologue -> recurrence -> epilogue
    run = dict(inp)
    for n in ("q", "k", "v"):
        run[n] = pkg.conv_silu(pre[n], cw[n]).view(B, T, N, -1)
    y, _ = pkg.m2rnn_forward(run)
    out = pkg.gate_rmsnorm(y.view(B, T, N * V), gpre, wn, 1e-6)
    assert pkg.stream_status() == binding.OK
    # oracle: the same stages in fp64, conv outputs rounded to bf16 as the GPU's are
    ref_in = all_f64(inp)
    for n in ("q", "k", "v"):
        c = conv_silu(pre[n].double().cpu().numpy(), cw[n].double().cpu().numpy())
        c = torch.from_numpy(c).to(torch.bfloat16).double().numpy()
        ref_in[n] = c.reshape(B, T, N, -1)
    yo, _ = m2rnn_forward_inputs(ref_in)
    # stage by stage: the readout at the recurrence's bar (3e-2), then the epilogue on the
    # GPU's own readout at the bf16 rounding bound (RMSNorm rescales any readout error by
    # |w SiLU(g)| / rms, so the chain's end-to-end bar is derived from these two)
    err_y = float(np.abs(y.double().cpu().numpy() - yo).max())
    assert err_y <= 3e-2, err_y
    ref = gate_rmsnorm(y.view(B, T, N * V).double().cpu().numpy(), gpre.double().cpu().numpy(),
                       wn.double().cpu().numpy(), 1e-6)
    assert close_bf16(out, ref) <= 0.0


def fused_case(B, T, N, K, V, shared=False, with_bias=True, seed=0, scale=1.5, tap=0.6):
    Nqk = 1 if shared else N
    wl = Workload("fz", B, T, N, K, V, h0="uniform", shared_qk=shared)
    inp = make_inputs(wl, DEV, seed)
    pre = {"q": rand_bf16((B, T, Nqk * K), seed + 1, scale),
           "k": rand_bf16((B, T, Nqk * K), seed + 2, scale),
           "v": rand_bf16((B, T, N * V), seed + 3, scale)}
    g = torch.Generator().manual_seed(seed + 4)
    conv = {}
    for n in ("q", "k", "v"):
        C = pre[n].shape[2]
        conv["w" + n] = (torch.randn((C, 4), generator=g) * tap).to(DEV)
        conv["b" + n] = (torch.randn(C, generator=g) * 0.1).to(DEV) if with_bias else None
    return inp, pre, conv, Nqk


@pytest.mark.parametrize("B,T,N,K,V,shared", [
    (2, 100, 3, 64, 64, False),   # ragged last chunk
    (1, 33, 2, 32, 16, False),
    (2, 2, 2, 64, 48, False),     # fewer steps than the conv window
    (2, 70, 4, 64, 64, True),     # q, k shared by the heads
    (8, 300, 16, 64, 64, False),  # 128 pairs: one block per pair
    (4, 200, 8, 64, 32, False),   # 32 pairs: two-block clusters
])
@pytest.mark.parametrize("with_bias", [True, False])
def test_fused_prologue_forward_is_bitwise_the_chain(B, T, N, K, V, shared, with_bias):
    """m2rnn_forward_conv gives the bits of conv_silu on each projection followed by the
    forward: the fused prologue runs the same fp32 operations and rounds to bf16 the same way."""
    inp, pre, conv, Nqk = fused_case(B, T, N, K, V, shared, with_bias, seed=B + T + K + V)
    run = dict(inp)
    for n in ("q", "k", "v"):
        run[n] = pkg.conv_silu(pre[n], conv["w" + n], conv["b" + n]).view(B, T, -1, V if n == "v" else K)
    y_ref, HT_ref = pkg.m2rnn_forward(run)
    fused_in = dict(inp)
    for n in ("q", "k", "v"):
        fused_in[n] = pre[n].view(B, T, -1, V if n == "v" else K)
    y, HT = pkg.m2rnn_forward_conv(fused_in, conv)
    assert pkg.stream_status() == binding.OK
    assert torch.equal(y, y_ref) and torch.equal(HT, HT_ref)


def test_fused_prologue_matches_oracle():
    """Against the fp64 oracle (conv outputs rounded to bf16 as the GPU's are), with the
    chained-block test's input scale (unit projections, taps of scale 0.5), at the
    recurrence's bf16 bar."""
    B, T, N, K, V = 2, 90, 3, 64, 64
    inp, pre, conv, _ = fused_case(B, T, N, K, V, seed=7, scale=1.0, tap=0.5)
    fused_in = dict(inp)
    for n in ("q", "k", "v"):
        fused_in[n] = pre[n].view(B, T, N, -1)
    y, HT = pkg.m2rnn_forward_conv(fused_in, conv)
    assert pkg.stream_status() == binding.OK
    ref_in = all_f64(inp)
    for n in ("q", "k", "v"):
        c = conv_silu(pre[n].double().cpu().numpy(), conv["w" + n].double().cpu().numpy(),
                      conv["b" + n].double().cpu().numpy())
        ref_in[n] = torch.from_numpy(c).to(torch.bfloat16).double().numpy().reshape(B, T, N, -1)
    yo, HTo = m2rnn_forward_inputs(ref_in)
    assert float(np.abs(y.double().cpu().numpy() - yo).max()) <= 3e-2
    assert float(np.abs(HT.double().cpu().numpy() - HTo).max()) <= 3e-2


def test_fused_prologue_unsupported_shape():
    inp, pre, conv, _ = fused_case(1, 10, 2, 128, 128, seed=3)
    fused_in = dict(inp)
    for n in ("q", "k", "v"):
        fused_in[n] = pre[n].view(1, 10, 2, -1)
    with pytest.raises(binding.M2RNNError) as e:
        pkg.m2rnn_forward_conv(fused_in, conv)
    assert e.value.status == binding.ERR_UNSUPPORTED
