"""Pins that tie the fp64 backward oracle to the forward definition and the notes.

Source: the M²RNN study notes ("M²RNN: 矩阵状态非线性 RNN 的容量、表达力与系统代价"),
Sec. 2.7 (chain-rule reverse scan) and Sec. 2.2 Eq. (13)/(17) (gate).  The pins
do not retype those formulas:
  * finite differences: for every input tensor, the directional derivative of a
    scalar loss L = <y, G_y> + <H_T, G_H> computed by central differences of the
    forward oracle (itself pinned in test_oracle_pins.py) must equal the inner
    product of the backward's gradient with the direction.  This checks every
    gradient against Eq. (10)-(13) directly, whatever formula produced it;
  * the same with one q, k set shared by all heads (Sec. 2.4, Sec. 2.7: shared
    q/k gradients add over heads);
  * hold (alpha = 0, so f = 1): the state never changes, so the gradient of H_0
    is dH_T + sum_t q_t u_t^T, and W, k get no gradient (a closed form that
    follows from Eq. (11) with f = 1);
  * T = 0: the only gradient is dH_0 = dH_T.
Every pin is a function of a ``backward`` callable, so the mutation test at the
bottom can check that each planted mistake in a copy of the oracle's arithmetic
(including the two pseudo-code slips the notes point out in Sec. 2.7) fails at
least one pin.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import scipy.special

from oracle import m2rnn_forward, softplus
from oracle.m2rnn_backward import m2rnn_backward, sigmoid

NAMES = ["q", "k", "v", "a", "alpha", "beta", "W", "w_r", "H0"]


def rand_problem(rng, B=2, T=6, N=2, K=3, V=4, shared=False, alpha=None):
    Nqk = 1 if shared else N
    p = dict(
        q=rng.normal(0, 1 / math.sqrt(K), (B, T, Nqk, K)),
        k=rng.normal(0, 1, (B, T, Nqk, K)),
        v=rng.normal(0, 1, (B, T, N, V)),
        a=rng.normal(0, 1, (B, T, N)),
        alpha=np.exp(rng.uniform(np.log(0.3), np.log(3.0), N)) if alpha is None else np.full(N, alpha),
        beta=rng.uniform(-2, 2, N),
        W=np.eye(V)[None] + rng.normal(0, math.sqrt(0.5 / V), (N, V, V)),
        w_r=rng.normal(0, 1, (N, V)),
        H0=rng.uniform(-0.5, 0.5, (B, N, K, V)),
    )
    Gy = rng.normal(0, 1, (B, T, N, V))
    GH = rng.normal(0, 1, (B, N, K, V))
    return p, Gy, GH


def loss(p, Gy, GH):
    y, HT = m2rnn_forward(p["q"], p["k"], p["v"], p["a"], p["alpha"], p["beta"], p["W"], p["w_r"],
                          p["H0"])
    return float(np.sum(y * Gy) + np.sum(HT * GH))


def grads(backward, p, Gy, GH):
    g = backward(p["q"], p["k"], p["v"], p["a"], p["alpha"], p["beta"], p["W"], p["w_r"], Gy,
                 p["H0"], GH)
    return {n: g["d" + n] for n in NAMES}


def fd_agrees(backward, p, Gy, GH, rng, eps=1e-5, rtol=1e-6):
    g = grads(backward, p, Gy, GH)
    for name in NAMES:
        d = rng.normal(0, 1, np.shape(p[name]))
        plus, minus = dict(p), dict(p)
        plus[name] = p[name] + eps * d
        minus[name] = p[name] - eps * d
        fd = (loss(plus, Gy, GH) - loss(minus, Gy, GH)) / (2 * eps)
        an = float(np.sum(np.asarray(g[name]) * d))
        if not abs(fd - an) <= rtol * max(1.0, abs(fd)):
            return False
    return True


# ---------------------------------------------------------------- pins
def pin_finite_differences(backward):
    rng = np.random.default_rng(11)
    return all(fd_agrees(backward, *rand_problem(rng), rng) for _ in range(2))


def pin_finite_differences_shared_qk(backward):
    rng = np.random.default_rng(12)
    return fd_agrees(backward, *rand_problem(rng, N=3, shared=True), rng)


def pin_finite_differences_long_saturated(backward):
    """Larger K, V and inputs large enough that tanh saturates on some elements."""
    rng = np.random.default_rng(13)
    p, Gy, GH = rand_problem(rng, B=1, T=9, N=1, K=5, V=6)
    p["k"] = p["k"] * 3.0
    return fd_agrees(backward, p, Gy, GH, rng)


def pin_hold(backward):
    rng = np.random.default_rng(14)
    p, Gy, GH = rand_problem(rng, alpha=0.0)
    g = grads(backward, p, Gy, GH)
    want_dH0 = GH + np.einsum("btnk,btnv->bnkv", p["q"], Gy)
    want_dq = np.einsum("bnkv,btnv->btnk", p["H0"], Gy)
    return (np.allclose(g["H0"], want_dH0, atol=1e-12) and np.allclose(g["q"], want_dq, atol=1e-12)
            and np.abs(g["W"]).max() == 0 and np.abs(g["k"]).max() == 0
            and np.abs(g["a"]).max() == 0 and np.abs(g["beta"]).max() == 0
            and np.allclose(g["v"], p["w_r"][None, None] * Gy, atol=1e-12))


def pin_empty_sequence(backward):
    rng = np.random.default_rng(15)
    p, Gy, GH = rand_problem(rng, T=0)
    g = grads(backward, p, Gy, GH)
    return (np.array_equal(g["H0"], GH) and np.abs(g["W"]).max() == 0
            and np.abs(g["alpha"]).max() == 0 and np.abs(g["w_r"]).max() == 0)


PINS = [pin_finite_differences, pin_finite_differences_shared_qk,
        pin_finite_differences_long_saturated, pin_hold, pin_empty_sequence]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_backward_oracle_pin(pin):
    assert pin(m2rnn_backward)


def test_sigmoid_is_stable_and_correct():
    x = np.array([-800.0, -30.0, -1.0, 0.0, 1.0, 30.0, 800.0])
    s = sigmoid(x)
    assert np.all(np.isfinite(s))
    assert np.allclose(s, scipy.special.expit(x), rtol=1e-15, atol=0)


# ---------------------------------------------------------------- mutation test
def _mutant(kind):
    """A copy of the backward oracle's arithmetic with one planted mistake."""
    def bwd(q, k, v, a, alpha, beta, W, w_r, dy, H0=None, dH_T=None):
        B, T, N, V = v.shape
        K = q.shape[-1]
        shared = q.shape[2] == 1 and N > 1
        qf = np.broadcast_to(q, (B, T, N, K))
        kf = np.broadcast_to(k, (B, T, N, K))
        _, _, states = m2rnn_forward(qf, kf, v, a, alpha, beta, W, w_r, H0, return_states=True)
        Hinit = np.zeros((B, N, K, V)) if H0 is None else H0
        x = a + beta
        f = np.exp(-alpha * softplus(x))
        C = np.zeros((B, N, K, V)) if dH_T is None else np.array(dH_T)
        dq, dk = np.empty((B, T, N, K)), np.empty((B, T, N, K))
        dv, df = np.empty((B, T, N, V)), np.empty((B, T, N))
        dW = np.zeros((N, V, V))
        Wt = np.swapaxes(W, -1, -2)
        for t in range(T - 1, -1, -1):
            Hp = states[:, t - 1] if t > 0 else Hinit
            Ht = states[:, t]
            u = dy[:, t]
            ft = f[:, t, :, None, None]
            Z = np.tanh(np.matmul(Hp, W) + kf[:, t, ..., :, None] * v[:, t, ..., None, :])
            R = C + qf[:, t, ..., :, None] * u[..., None, :]
            if kind == "no_carry":               # readout term only, future gradient dropped
                R = qf[:, t, ..., :, None] * u[..., None, :]
            dtanh = 1 - Z if kind == "dtanh_wrong" else 1 - Z * Z
            D = ((1 - ft) * R) * dtanh
            df[:, t] = np.einsum("bnkv,bnkv->bn", R, (Z - Hp) if kind == "df_sign" else (Hp - Z))
            dW += np.einsum("bnki,bnkj->nji" if kind == "dW_transposed" else "bnki,bnkj->nij", Hp, D)
            dk[:, t] = np.einsum("bnkv,bnv->bnk", D, v[:, t])
            dv[:, t] = np.einsum("bnkv,bnk->bnv", D, kf[:, t])
            if kind != "dv_no_residual":
                dv[:, t] += w_r[None] * u
            dq[:, t] = np.einsum("bnkv,bnv->bnk", Hp if kind == "dq_prev_state" else Ht, u)
            prop = D @ (W if kind == "W_not_transposed" else Wt)
            C = prop if kind == "no_retain" else ft * R + prop   # retained branch dropped
        sx = sigmoid(-x) if kind == "gate_sigmoid_sign" else sigmoid(x)
        da = df * (-alpha * f * sx)
        dalpha = np.einsum("btn->n", df * (-f * softplus(x)))
        dbeta = np.einsum("btn->n", da)
        dw_r = np.einsum("btnv,btnv->nv", dy, v)
        if shared and kind != "shared_not_summed":
            dq, dk = dq.sum(2, keepdims=True), dk.sum(2, keepdims=True)
        elif shared:
            dq, dk = dq[:, :, :1], dk[:, :, :1]
        return {"dq": dq, "dk": dk, "dv": dv, "da": da, "dalpha": dalpha, "dbeta": dbeta,
                "dW": dW, "dw_r": dw_r, "dH0": C}
    return bwd


MUTANTS = ["no_carry", "no_retain", "W_not_transposed", "dtanh_wrong", "df_sign", "dW_transposed",
           "dv_no_residual", "dq_prev_state", "gate_sigmoid_sign", "shared_not_summed"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_each_planted_mistake_fails_a_pin(kind):
    bwd = _mutant(kind)
    assert not all(pin(bwd) for pin in PINS), f"mutant {kind} passes every pin"


def test_unmutated_copy_passes_all_pins():
    bwd = _mutant("none")
    assert all(pin(bwd) for pin in PINS)
