"""Multi-value sharing (one q, k set for all heads; the M²RNN notes' Sec. 2.4, N_q = N_k = 1).

CPU: the oracle with q, k of shape [B, T, 1, K] equals the oracle with those vectors
tiled over the N heads (bitwise: the same arithmetic), the scalar brute force agrees,
and the C ABI rejects a q/k head count other than 1 or N before launching anything.
"""
import numpy as np
import pytest

import __graft_entry__
from matrix_state_nonlinear_gb300 import m2rnn as binding
from oracle import m2rnn_forward, m2rnn_forward_scalar


def shared_problem(rng, B, T, N, K, V):
    q = rng.normal(0, 1 / np.sqrt(K), (B, T, 1, K))
    k = rng.normal(0, 1 / np.sqrt(K), (B, T, 1, K))
    v = rng.normal(0, 1, (B, T, N, V))
    a = rng.normal(0, 1, (B, T, N))
    al = np.exp(rng.uniform(np.log(0.3), np.log(3.0), N))
    be = rng.uniform(-2, 2, N)
    W = np.eye(V)[None] + rng.normal(0, np.sqrt(0.3 / V), (N, V, V))
    w_r = rng.normal(0, 1, (N, V))
    H0 = rng.uniform(-0.5, 0.5, (B, N, K, V))
    return q, k, v, a, al, be, W, w_r, H0


def test_shared_equals_tiled_per_head_bitwise():
    q, k, v, a, al, be, W, w_r, H0 = shared_problem(np.random.default_rng(21), 2, 9, 3, 4, 5)
    ys, Hs = m2rnn_forward(q, k, v, a, al, be, W, w_r, H0)
    qt, kt = np.repeat(q, 3, axis=2), np.repeat(k, 3, axis=2)
    yt, Ht = m2rnn_forward(qt, kt, v, a, al, be, W, w_r, H0)
    assert np.array_equal(ys, yt) and np.array_equal(Hs, Ht)


def test_shared_agrees_with_scalar_brute_force():
    q, k, v, a, al, be, W, w_r, H0 = shared_problem(np.random.default_rng(22), 1, 4, 3, 2, 3)
    y, H = m2rnn_forward(q, k, v, a, al, be, W, w_r, H0)
    ys, Hs = m2rnn_forward_scalar(q, k, v, a, al, be, W, w_r, H0)
    np.testing.assert_allclose(y, ys, rtol=0, atol=1e-12)
    np.testing.assert_allclose(H, Hs, rtol=0, atol=1e-12)


def test_heads_differ_only_through_v_f_W():
    # With shared q, k, two heads with identical v, gate and W give identical outputs.
    q, k, v, a, al, be, W, w_r, H0 = shared_problem(np.random.default_rng(23), 1, 6, 2, 3, 3)
    v[:, :, 1], a[:, :, 1], al[1], be[1], W[1], w_r[1] = v[:, :, 0], a[:, :, 0], al[0], be[0], W[0], w_r[0]
    H0[:, 1] = H0[:, 0]
    y, H = m2rnn_forward(q, k, v, a, al, be, W, w_r, H0)
    assert np.array_equal(y[:, :, 0], y[:, :, 1]) and np.array_equal(H[:, 0], H[:, 1])


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return binding.load_library()


@pytest.mark.parametrize("Nqk", [0, 2, 5])
def test_bad_qk_head_count_is_invalid_arg(lib, Nqk):
    p = [(1 << 20) + 256 * i for i in range(11)]
    assert lib.m2rnn_forward_f32_qk(*p, 1, 4, 3, Nqk, 8, 8, None) == binding.ERR_INVALID_ARG
    assert lib.m2rnn_forward_bf16_qk(*p, 1, 4, 3, Nqk, 16, 16, 0, None) == binding.ERR_INVALID_ARG
