"""The seeded generator (determinism, shapes, distributions) and the frozen oracle fixture."""
import json
import math
import os

import numpy as np
import torch

from matrix_state_nonlinear_gb300.inputs import (WORKLOADS, all_f64, make_inputs, make_params,
                                                 slice_pair)
from oracle import m2rnn_forward, m2rnn_forward_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_f32_b1_t64_n2_k8_v8.json")


def small(name="b4_t2048_n8_k64_v64", **kw):
    return WORKLOADS[name].with_(**kw)


def test_same_seed_same_bits_and_shapes():
    wl = small(T=33, B=2, N=3)
    a, b = make_inputs(wl, "cpu", 0), make_inputs(wl, "cpu", 0)
    c = make_inputs(wl, "cpu", 1)
    for key in a:
        if a[key] is None:
            continue
        assert torch.equal(a[key], b[key])
    assert not torch.equal(a["q"], c["q"])
    assert a["q"].shape == (2, 33, 3, 64) and a["v"].shape == (2, 33, 3, 64)
    assert a["a"].shape == (2, 33, 3) and a["W"].shape == (3, 64, 64)
    assert a["q"].dtype == torch.bfloat16 and a["alpha"].dtype == torch.float32
    assert all(t.is_contiguous() for t in a.values() if t is not None)


def test_distributions():
    wl = small(T=512, B=2, N=8)
    inp = make_inputs(wl, "cpu", 0)
    q = inp["q"].float()
    assert abs(q.std().item() - 1 / math.sqrt(64)) < 0.01
    assert abs(inp["v"].float().std().item() - 1.0) < 0.02
    al = inp["alpha"].numpy()
    assert np.all((al >= 0.5) & (al <= 2.0))
    be = inp["beta"].numpy()
    assert np.all((be >= -2) & (be <= 2))
    W = inp["W"].double().numpy()
    for n in range(wl.N):
        s = np.linalg.svd(W[n], compute_uv=False)[0]
        assert s <= 1.0 + 2 ** -7
    wide = WORKLOADS["b16_t8192_n32_k128_v128"].with_(B=2, T=4, N=4)
    p = make_params(wide)
    assert p["H0"].shape == (2, 4, 128, 128) and np.all(np.abs(p["H0"]) <= 0.5)
    assert np.all((p["alpha"] >= 0.1) & (p["alpha"] <= 4.0))


def test_pair_slice_matches_full_problem():
    wl = small(T=40, B=2, N=3, K=16, V=16, h0="uniform")
    inp = make_inputs(wl, "cpu", 0)
    y, HT = m2rnn_forward_inputs(all_f64(inp))
    ys, HTs = m2rnn_forward_inputs(slice_pair(inp, 1, 2))
    np.testing.assert_allclose(ys[0, :, 0], y[1, :, 2], rtol=0, atol=1e-13)
    np.testing.assert_allclose(HTs[0, 0], HT[1, 2], rtol=0, atol=1e-13)


def test_golden_fixture_reproduces():
    doc = json.load(open(GOLDEN))
    s = doc["shape"]
    B, T, N, K, V = s["B"], s["T"], s["N"], s["K"], s["V"]
    i = doc["inputs"]
    arr = lambda key, shp: np.array(i[key], dtype=np.float64).reshape(shp)
    y, HT = m2rnn_forward(arr("q", (B, T, N, K)), arr("k", (B, T, N, K)), arr("v", (B, T, N, V)),
                          arr("a", (B, T, N)), arr("alpha", (N,)), arr("beta", (N,)),
                          arr("W", (N, V, V)), arr("w_r", (N, V)), None)
    np.testing.assert_allclose(y.ravel(), np.array(doc["y"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(HT.ravel(), np.array(doc["H_T"]), rtol=0, atol=1e-13)
    # the stored inputs are the generator's current output
    gen = all_f64(make_inputs(WORKLOADS[doc["workload"]], "cpu", 0))
    np.testing.assert_array_equal(gen["q"].ravel(), np.array(i["q"]))
