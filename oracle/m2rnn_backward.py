"""fp64 CPU oracle for the M²RNN backward pass.  TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The CUDA library never calls it and shares
no code with it.

Source: the M²RNN study notes ("M²RNN: 矩阵状态非线性 RNN 的容量、表达力与系统代价"):
  * Sec. 2.6 (the paper's Sec. 4.2): the backward re-runs the recurrence, keeps
    every step's state, then scans time in reverse.
  * Sec. 2.7: the chain-rule form of the reverse scan, with u_t = dL/d(H_t^T q_t)
    and C_t the state gradient arriving from later steps:
        R_t     = C_t + q_t u_t^T
        D_t     = ((1 - f_t) R_t) ⊙ (1 - Z_t ⊙ Z_t)
        C_{t-1} = f_t R_t + D_t W^T
        dL/df_t = <R_t, H_{t-1} - Z_t>_F,   dL/dW = sum_t H_{t-1}^T D_t,
        dL/dk_t = D_t v_t,  dL/dv_t = D_t^T k_t (+ w_r ⊙ u_t),  dL/dq_t = H_t u_t.
    Shared q/k gradients add over heads; W gradients add over batch and time.
  * Sec. 2.2, Eq. (13)/(17), differentiated: with x = a + beta and
    f = exp(-alpha softplus(x)),
        df/da = df/dbeta = -alpha f sigmoid(x),   df/dalpha = -f softplus(x).
  * Eq. (12): the direct path y_t ∋ w_r ⊙ v_t gives dL/dw_r = sum_t u_t ⊙ v_t.

Readings taken where the notes leave a step open:
  * The loss reaches the recurrence through y (gradient dy = u) and through the
    final state H_T (gradient dH_T, zero when absent); C_T = dH_T.
  * The gradient of the initial state is C_{-1} after the last reverse step (dH_0).
  * Z_t is recomputed from the kept H_{t-1} (Sec. 2.6 keeps states, not Z).

The reverse scan is written out one time step after another in fp64, vectorised
only over the independent (batch, head) pairs, in the notes' order.  Its pins
(finite differences of the forward oracle, closed forms) are in
tests/test_backward_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np

from .m2rnn_oracle import m2rnn_forward, softplus


def sigmoid(x):
    x = np.asarray(x, np.float64)
    return np.where(x >= 0, 1.0 / (1.0 + np.exp(-np.abs(x))),
                    np.exp(-np.abs(x)) / (1.0 + np.exp(-np.abs(x))))


def m2rnn_backward(q, k, v, a, alpha, beta, W, w_r, dy, H0=None, dH_T=None):
    """Gradients of L(y, H_T) given dy = dL/dy [B,T,N,V] and dH_T = dL/dH_T [B,N,K,V].

    Inputs as for ``m2rnn_forward`` (q, k may be [B,T,1,K]: shared by all heads).
    Returns a dict with dq, dk (shaped like q, k), dv [B,T,N,V], da [B,T,N],
    dalpha [N], dbeta [N], dW [N,V,V], dw_r [N,V], dH0 [B,N,K,V].
    """
    v = np.asarray(v, np.float64)
    a = np.asarray(a, np.float64)
    alpha = np.asarray(alpha, np.float64)
    beta = np.asarray(beta, np.float64)
    W = np.asarray(W, np.float64)
    w_r = np.asarray(w_r, np.float64)
    dy = np.asarray(dy, np.float64)
    B, T, N, V = v.shape
    K = np.shape(q)[-1]
    shared = np.shape(q)[2] == 1 and N > 1
    qf = np.broadcast_to(np.asarray(q, np.float64), (B, T, N, K))
    kf = np.broadcast_to(np.asarray(k, np.float64), (B, T, N, K))

    # Re-run the recurrence and keep every state (Sec. 2.6).
    _, _, states = m2rnn_forward(qf, kf, v, a, alpha, beta, W, w_r, H0, return_states=True)
    Hinit = np.zeros((B, N, K, V)) if H0 is None else np.asarray(H0, np.float64)

    x = a + beta                                          # [B,T,N]
    f = np.exp(-alpha * softplus(x))                      # Eq. (13)/(17)

    C = np.zeros((B, N, K, V)) if dH_T is None else np.array(dH_T, dtype=np.float64)
    dq = np.empty((B, T, N, K))
    dk = np.empty((B, T, N, K))
    dv = np.empty((B, T, N, V))
    df = np.empty((B, T, N))
    dW = np.zeros((N, V, V))
    for t in range(T - 1, -1, -1):
        H_prev = states[:, t - 1] if t > 0 else Hinit     # H_{t-1}
        H_t = states[:, t]
        u = dy[:, t]                                      # [B,N,V]
        qt, kt, vt = qf[:, t], kf[:, t], v[:, t]
        ft = f[:, t, :, None, None]
        Z = np.tanh(np.matmul(H_prev, W) + kt[..., :, None] * vt[..., None, :])   # Eq. (10)
        R = C + qt[..., :, None] * u[..., None, :]        # R_t = C_t + q_t u_t^T
        D = ((1.0 - ft) * R) * (1.0 - Z * Z)              # D_t
        df[:, t] = np.einsum("bnkv,bnkv->bn", R, H_prev - Z)
        dW += np.einsum("bnki,bnkj->nij", H_prev, D)      # sum over b of H_{t-1}^T D_t
        dk[:, t] = np.einsum("bnkv,bnv->bnk", D, vt)      # D_t v_t
        dv[:, t] = np.einsum("bnkv,bnk->bnv", D, kt) + w_r[None] * u   # D_t^T k_t + w_r ⊙ u_t
        dq[:, t] = np.einsum("bnkv,bnv->bnk", H_t, u)     # H_t u_t
        C = ft * R + np.matmul(D, np.swapaxes(W, -1, -2))  # C_{t-1} = f_t R_t + D_t W^T

    # Gate parameters through Eq. (13)/(17).
    da = df * (-alpha * f * sigmoid(x))
    dalpha = np.einsum("btn->n", df * (-f * softplus(x)))
    dbeta = np.einsum("btn->n", da)
    dw_r = np.einsum("btnv,btnv->nv", dy, v)
    if shared:  # one q_t, k_t for every head: their gradients add over heads (Sec. 2.7)
        dq = dq.sum(axis=2, keepdims=True)
        dk = dk.sum(axis=2, keepdims=True)
    return {"dq": dq, "dk": dk, "dv": dv, "da": da, "dalpha": dalpha, "dbeta": dbeta,
            "dW": dW, "dw_r": dw_r, "dH0": C}


def m2rnn_backward_inputs(inp: dict, dy, dH_T=None):
    """``m2rnn_backward`` on a dict of fp64 arrays keyed like the input generator's."""
    return m2rnn_backward(inp["q"], inp["k"], inp["v"], inp["a"], inp["alpha"], inp["beta"],
                          inp["W"], inp["w_r"], dy, inp.get("H0"), dH_T)
