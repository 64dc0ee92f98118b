"""Pins that tie the fp64 oracle to what the M²RNN notes and mathematics fix.

Source: the M²RNN study notes ("M²RNN: 矩阵状态非线性 RNN 的容量、表达力与系统代价",
on arXiv:2603.14360v2).  Each pin names the passage it follows:
  * gate, Sec. 2.2 Eq. (13)/(17): alpha = 1 gives sigma(-a - beta); the two
    printed forms agree; alpha = 0 gives f = 1;
  * hold, Sec. 2.1 (reading of Eq. (11)): f = 1 keeps the state;
  * W = 0: Eq. (10)-(11) become an elementwise linear recurrence with a
    closed-form sum;
  * Theorem 1 / App. B Eq. (25) (Sec. 2.5): f = 0, w_r = 0, q = k = e_1 turn the
    first row into the tanh RNN h_t = tanh(W^T h_{t-1} + v_t), checked against
    torch.nn.RNN;
  * boundedness, Sec. 2.1: H_0 = 0 and f in [0, 1] keep |H| <= 1;
  * readout, Eq. (12): linear in w_r; |y - w_r v| <= ||q||_1;
  * rows of H are independent given W and f (Sec. 1.2: W mixes value dims,
    not key rows), so a row permutation of (H_0, k, q) leaves y unchanged;
  * state carry: chunked == full; prefix causality;
  * brute force: pure-Python scalar loops on tiny shapes.
Every pin is a function of a ``forward`` callable, so the mutation test at the
bottom can check that each planted mistake in a copy of the oracle's arithmetic
fails at least one pin.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import scipy.special
import torch

from oracle import forget_gate, m2rnn_forward, m2rnn_forward_scalar, softplus


def rand_problem(rng, B, T, N, K, V, h0=True, alpha=None, scale=1.0):
    q = rng.normal(0, 1 / math.sqrt(K), (B, T, N, K))
    k = rng.normal(0, 1 / math.sqrt(K), (B, T, N, K)) * scale
    v = rng.normal(0, 1, (B, T, N, V)) * scale
    a = rng.normal(0, 1, (B, T, N))
    al = np.exp(rng.uniform(np.log(0.3), np.log(3.0), N)) if alpha is None else np.full(N, alpha)
    be = rng.uniform(-2, 2, N)
    W = np.eye(V)[None] + rng.normal(0, math.sqrt(0.3 / V), (N, V, V))
    w_r = rng.normal(0, 1, (N, V))
    H0 = rng.uniform(-0.5, 0.5, (B, N, K, V)) if h0 else None
    return dict(q=q, k=k, v=v, a=a, alpha=al, beta=be, W=W, w_r=w_r, H0=H0)


def run(forward, p, **over):
    d = dict(p)
    d.update(over)
    return forward(d["q"], d["k"], d["v"], d["a"], d["alpha"], d["beta"], d["W"], d["w_r"],
                   d["H0"])


# ---------------------------------------------------------------- gate pins (Eq. 13/17)
def test_gate_alpha_one_is_sigmoid():
    rng = np.random.default_rng(1)
    a = rng.normal(0, 3, (50, 4))
    beta = rng.uniform(-2, 2, 4)
    f = forget_gate(a, np.ones(4), beta)
    np.testing.assert_allclose(f, scipy.special.expit(-(a + beta)), rtol=1e-14, atol=0)


def test_gate_printed_forms_agree():
    # Eq. (13) prints (1 + e^{a+beta})^{-alpha}; Eq. (17) exp(-alpha softplus(a+beta)).
    rng = np.random.default_rng(2)
    a = rng.normal(0, 2, (40, 3))
    alpha = np.array([0.1, 1.7, 4.0])
    beta = np.array([-1.5, 0.3, 2.0])
    direct = np.power(1.0 + np.exp(a + beta), -alpha)
    np.testing.assert_allclose(forget_gate(a, alpha, beta), direct, rtol=1e-13)


def test_gate_alpha_zero_is_one_and_range():
    a = np.linspace(-800, 800, 101)[:, None]
    f0 = forget_gate(a, np.zeros(1), np.zeros(1))
    assert np.all(f0 == 1.0)
    f = forget_gate(a, np.full(1, 2.5), np.full(1, 0.7))
    assert np.all(np.isfinite(f)) and np.all((f >= 0) & (f <= 1))
    # softplus must not overflow and must match log(1+e^x) where that is representable
    x = np.array([-700.0, -30.0, -1.0, 0.0, 1.0, 30.0, 700.0])
    sp = softplus(x)
    assert np.all(np.isfinite(sp))
    np.testing.assert_allclose(sp[1:6], np.log1p(np.exp(x[1:6])), rtol=1e-15)
    assert sp[-1] == 700.0


# ---------------------------------------------------------------- pin functions
def pin_hold(forward):
    """alpha = 0 => f = 1 => H_t = H_0 for all t; y_t = H_0^T q_t + w_r ⊙ v_t."""
    p = rand_problem(np.random.default_rng(3), 2, 9, 3, 4, 5, h0=True, alpha=0.0)
    y, HT = run(forward, p)
    if not np.array_equal(HT, p["H0"]):
        return False
    expect = np.einsum("bnkv,btnk->btnv", p["H0"], p["q"]) + p["w_r"][None, None] * p["v"]
    return np.allclose(y, expect, rtol=0, atol=1e-12)


def pin_w_zero_closed_form(forward):
    """W = 0: H_T = (prod_s f_s) H_0 + sum_s (1-f_s) (prod_{r>s} f_r) tanh(k_s v_s^T)."""
    rng = np.random.default_rng(4)
    B, T, N, K, V = 2, 7, 2, 3, 4
    p = rand_problem(rng, B, T, N, K, V, h0=True)
    p["W"] = np.zeros((N, V, V))
    y, HT = run(forward, p)
    sig = 1.0 / (1.0 + np.exp(p["a"] + p["beta"]))           # sigma(-(a+beta))
    f = sig ** p["alpha"]                                     # Eq. (13) form
    ok = True
    for b in range(B):
        for n in range(N):
            for tt in range(T):                               # state after step tt
                Ht = np.prod(f[b, :tt + 1, n]) * p["H0"][b, n]
                for s in range(tt + 1):
                    tail = np.prod(f[b, s + 1:tt + 1, n])
                    Ht = Ht + (1 - f[b, s, n]) * tail * np.tanh(np.outer(p["k"][b, s, n],
                                                                          p["v"][b, s, n]))
                ys = Ht.T @ p["q"][b, tt, n] + p["w_r"][n] * p["v"][b, tt, n]
                ok &= np.allclose(ys, y[b, tt, n], rtol=0, atol=1e-12)
            ok &= np.allclose(Ht, HT[b, n], rtol=0, atol=1e-12)
    return bool(ok)


def pin_f_zero_w_zero(forward):
    """f -> 0 and W = 0: H_t = tanh(k_t v_t^T) exactly, y_t = H_t^T q_t + w_r ⊙ v_t."""
    rng = np.random.default_rng(5)
    B, T, N, K, V = 1, 5, 2, 3, 3
    p = rand_problem(rng, B, T, N, K, V, h0=True)
    p.update(W=np.zeros((N, V, V)), alpha=np.full(N, 100.0), beta=np.full(N, 8.0),
             a=np.abs(p["a"]))                                  # a + beta >= 8: f < e^-800
    y, HT = run(forward, p)
    Hs = np.tanh(p["k"][..., :, None] * p["v"][..., None, :])  # [B,T,N,K,V]
    expect = np.einsum("btnkv,btnk->btnv", Hs, p["q"]) + p["w_r"][None, None] * p["v"]
    return np.allclose(y, expect, atol=1e-12) and np.allclose(HT, Hs[:, -1], atol=1e-12)


def pin_theorem1_vector_rnn(forward):
    """Theorem 1: f = 0, w_r = 0, q = k = e_1, H_0 = 0 => row 1 is a tanh RNN.

    h_t = tanh(W^T h_{t-1} + v_t) is torch.nn.RNN with W_ih = I, W_hh = W^T and
    no bias; the other rows of H stay zero and y_t = h_t.
    """
    rng = np.random.default_rng(6)
    B, T, N, K, V = 2, 12, 2, 3, 5
    p = rand_problem(rng, B, T, N, K, V, h0=False)
    e1 = np.zeros(K)
    e1[0] = 1.0
    p.update(q=np.broadcast_to(e1, (B, T, N, K)).copy(), k=np.broadcast_to(e1, (B, T, N, K)).copy(),
             w_r=np.zeros((N, V)), alpha=np.full(N, 100.0), beta=np.full(N, 6.0),
             a=np.abs(p["a"]), H0=None)
    y, HT = run(forward, p)
    ok = bool(np.all(HT[:, :, 1:, :] == 0.0))
    for n in range(N):
        rnn = torch.nn.RNN(V, V, nonlinearity="tanh", bias=False, batch_first=True,
                           dtype=torch.float64)
        with torch.no_grad():
            rnn.weight_ih_l0.copy_(torch.eye(V, dtype=torch.float64))
            rnn.weight_hh_l0.copy_(torch.tensor(p["W"][n].T))
            out, _ = rnn(torch.tensor(p["v"][:, :, n, :]))
        ok &= np.allclose(y[:, :, n, :], out.numpy(), rtol=0, atol=1e-12)
    return bool(ok)


def pin_bounded(forward):
    """H_0 = 0 and f in [0, 1] => every |H_t| <= 1 (convex combination of bounded terms)."""
    rng = np.random.default_rng(7)
    p = rand_problem(rng, 2, 40, 2, 3, 4, h0=False, scale=6.0)
    p["W"] = p["W"] * 3.0
    p["alpha"] = np.array([0.05, 5.0])
    ok = True
    for t in (1, 5, 40):
        sub = {kk: (vv[:, :t] if kk in ("q", "k", "v", "a") else vv) for kk, vv in p.items()}
        _, HT = run(forward, sub)
        ok &= bool(np.max(np.abs(HT)) <= 1.0)
    # the state must actually move: a vacuous zero state would pass the bound trivially
    return ok and float(np.max(np.abs(HT))) > 0.5


def pin_readout(forward):
    """Eq. (12): y is affine in w_r with slope v; |y_t - w_r ⊙ v_t| <= ||q_t||_1 when |H| <= 1."""
    rng = np.random.default_rng(8)
    p = rand_problem(rng, 2, 10, 2, 4, 3, h0=False)
    y1, _ = run(forward, p)
    y0, _ = run(forward, p, w_r=np.zeros_like(p["w_r"]))
    ok = np.allclose(y1 - y0, p["w_r"][None, None] * p["v"], rtol=0, atol=1e-12)
    bound = np.abs(p["q"]).sum(-1)[..., None]
    ok &= bool(np.all(np.abs(y0) <= bound + 1e-12))
    # the readout sums over K rows: q = e_i picks out H_t[i, :]
    p2 = dict(p)
    qe = np.zeros_like(p["q"])
    qe[..., 2] = 1.0
    p2["q"] = qe
    y2, HT2 = run(forward, p2, w_r=np.zeros_like(p["w_r"]))
    ok &= np.allclose(y2[:, -1], HT2[:, :, 2, :], atol=1e-12)
    return bool(ok)


def pin_row_permutation(forward):
    """Rows evolve independently: permuting rows of (H_0, k, q) leaves y unchanged."""
    rng = np.random.default_rng(9)
    p = rand_problem(rng, 2, 8, 2, 5, 4, h0=True)
    perm = np.array([3, 0, 4, 1, 2])
    y, HT = run(forward, p)
    yp, HTp = run(forward, p, q=p["q"][..., perm], k=p["k"][..., perm], H0=p["H0"][:, :, perm])
    return np.allclose(y, yp, atol=1e-12) and np.allclose(HT[:, :, perm], HTp, atol=1e-13)


def pin_zero_rows_stay_zero(forward):
    """A row with k_{t,i} = 0 for all t and a zero H_0 row stays zero."""
    rng = np.random.default_rng(10)
    p = rand_problem(rng, 1, 9, 2, 4, 3, h0=True)
    p["k"][..., 1] = 0.0
    p["H0"][:, :, 1, :] = 0.0
    _, HT = run(forward, p)
    return bool(np.all(HT[:, :, 1, :] == 0.0)) and bool(np.any(HT[:, :, 0, :] != 0.0))


def pin_brute_force(forward):
    """Agreement with nested scalar loops written from Eq. (10)-(13) on tiny shapes."""
    rng = np.random.default_rng(11)
    ok = True
    for (B, T, N, K, V) in [(1, 3, 1, 1, 1), (2, 4, 2, 2, 3), (1, 5, 2, 3, 2), (2, 3, 1, 4, 4)]:
        for h0 in (False, True):
            p = rand_problem(rng, B, T, N, K, V, h0=h0, scale=1.5)
            y, HT = run(forward, p)
            ys, HTs = run(m2rnn_forward_scalar, p)
            ok &= np.allclose(y, ys, rtol=0, atol=1e-12) and np.allclose(HT, HTs, rtol=0, atol=1e-12)
    return bool(ok)


PINS = [pin_hold, pin_w_zero_closed_form, pin_f_zero_w_zero, pin_theorem1_vector_rnn,
        pin_bounded, pin_readout, pin_row_permutation, pin_zero_rows_stay_zero, pin_brute_force]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    assert pin(m2rnn_forward)


# ---------------------------------------------------------------- state carry
def test_chunked_equals_full_bitwise():
    p = rand_problem(np.random.default_rng(12), 2, 20, 3, 4, 5, h0=True)
    y, HT = run(m2rnn_forward, p)
    cut = {kk: vv[:, :7] if kk in ("q", "k", "v", "a") else vv for kk, vv in p.items()}
    rest = {kk: vv[:, 7:] if kk in ("q", "k", "v", "a") else vv for kk, vv in p.items()}
    y1, H1 = run(m2rnn_forward, cut)
    rest["H0"] = H1
    y2, H2 = run(m2rnn_forward, rest)
    assert np.array_equal(np.concatenate([y1, y2], axis=1), y) and np.array_equal(H2, HT)


def test_prefix_causality_bitwise():
    p = rand_problem(np.random.default_rng(13), 2, 16, 2, 3, 4, h0=True)
    y, _ = run(m2rnn_forward, p)
    p2 = {kk: (vv.copy() if isinstance(vv, np.ndarray) else vv) for kk, vv in p.items()}
    for key in ("q", "k", "v", "a"):
        p2[key][:, 9:] += 1.0
    y2, _ = run(m2rnn_forward, p2)
    assert np.array_equal(y[:, :9], y2[:, :9]) and not np.allclose(y[:, 9:], y2[:, 9:])


def test_T_zero_returns_initial_state():
    p = rand_problem(np.random.default_rng(14), 1, 0, 2, 3, 4, h0=True)
    y, HT = run(m2rnn_forward, p)
    assert y.shape == (1, 0, 2, 4) and np.array_equal(HT, p["H0"])
    p["H0"] = None
    _, HT0 = run(m2rnn_forward, p)
    assert np.array_equal(HT0, np.zeros((1, 2, 3, 4)))


# ---------------------------------------------------------------- mutation test
def _mutant(kind):
    """A copy of the oracle's arithmetic with one planted mistake."""
    def fwd(q, k, v, a, alpha, beta, W, w_r, H0=None):
        B, T, N, K = q.shape
        V = v.shape[-1]
        H = np.zeros((B, N, K, V)) if H0 is None else np.array(H0, dtype=np.float64)
        x = a + beta
        if kind == "gate_sign":
            x = a - beta
        f = np.exp(-alpha * softplus(x))
        if kind == "gate_alpha_outside":
            f = np.exp(-softplus(alpha * x))
        y = np.empty((B, T, N, V))
        for t in range(T):
            Wm = np.swapaxes(W, -1, -2) if kind == "w_transposed" else W
            kv = k[:, t, :, :, None] * v[:, t, :, None, :]
            if kind == "no_rank1":
                kv = 0 * kv
            Z = np.tanh(np.matmul(H, Wm) + kv)
            if kind == "rank1_outside_tanh":
                Z = np.tanh(np.matmul(H, Wm)) + kv
            ft = f[:, t, :, None, None]
            Hn = ft * H + (1 - ft) * Z
            if kind == "swap_lerp":
                Hn = (1 - ft) * H + ft * Z
            Hr = H if kind == "readout_before_update" else Hn
            y[:, t] = np.einsum("bnkv,bnk->bnv", Hr, q[:, t]) + w_r[None] * v[:, t]
            if kind == "no_residual":
                y[:, t] -= w_r[None] * v[:, t]
            if kind == "readout_k":
                y[:, t] = np.einsum("bnkv,bnk->bnv", Hr, k[:, t]) + w_r[None] * v[:, t]
            H = Hn
        return y, H
    return fwd


MUTANTS = ["gate_sign", "gate_alpha_outside", "w_transposed", "no_rank1", "rank1_outside_tanh",
           "swap_lerp", "readout_before_update", "no_residual", "readout_k"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_each_planted_mistake_fails_a_pin(kind):
    fwd = _mutant(kind)
    assert not all(pin(fwd) for pin in PINS), f"mutant {kind} passes every pin"


def test_unmutated_copy_passes_all_pins():
    fwd = _mutant("none")
    assert all(pin(fwd) for pin in PINS)
