"""fp64 CPU oracle for the M²RNN forward recurrence.  TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The CUDA library never calls it and shares
no code with it.

Source: the M²RNN study notes ("M²RNN: 矩阵状态非线性 RNN 的容量、表达力与系统代价",
notes on Mishra, Tan, Stoica, Gonzalez, Dao, arXiv:2603.14360v2):
  * Sec. 2.1, Eq. (10)-(12), starting from H_0 = 0:
        Z_t = tanh(H_{t-1} W + k_t v_t^T)
        H_t = f_t H_{t-1} + (1 - f_t) Z_t
        y_t = H_t^T q_t + w_r ⊙ v_t
  * Sec. 2.2, Eq. (13)/(17): f_{t,n} = (1 + e^{a_{t,n} + beta_n})^{-alpha_n}
                                   = exp(-alpha_n softplus(a_{t,n} + beta_n))
  * Sec. 2.6 (Sec. 4.1 of the paper): each (batch, head) pair is an independent
    unit; time is processed in order.

Readings taken where the notes leave a step open:
  * f is one scalar per (b, t, n), broadcast over the K x V state (symbol table).
  * The readout uses H_t, the state after the update (Eq. 12 names H_t).
  * q, k are per head, [B, T, N, K]; W is per head and right-multiplied,
    (H W)_{ij} = sum_l H_{il} W_{lj}; w_r is per head, [N, V].
  * softplus is the exact log(1 + e^x), evaluated in its overflow-free form
    max(x, 0) + log1p(exp(-|x|)); no threshold linearisation.
  * An absent H_0 means the zero state.

The method has no approximation: the oracle is the definition written out in
fp64, one time step after another, vectorised only over the independent
(batch, head) pairs.  Pins that tie it to the notes rather than to itself are
in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import math

import numpy as np


def softplus(x: np.ndarray) -> np.ndarray:
    """log(1 + e^x) without overflow (the softplus of Eq. (17))."""
    x = np.asarray(x, dtype=np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def forget_gate(a: np.ndarray, alpha: np.ndarray, beta: np.ndarray) -> np.ndarray:
    """f = exp(-alpha * softplus(a + beta)), Eq. (13)/(17).

    a: [..., N] gate logits (the head axis last); alpha, beta: [N].
    """
    return np.exp(-np.asarray(alpha, np.float64) * softplus(np.asarray(a, np.float64) + beta))


def m2rnn_forward(q, k, v, a, alpha, beta, W, w_r, H0=None, return_states=False):
    """The forward recurrence over all (batch, head) pairs, in fp64.

    Shapes (row-major): q, k [B,T,N,K], or [B,T,1,K] when one query/key set is shared
    by all heads (Sec. 2.4); v [B,T,N,V]; a [B,T,N]; alpha, beta [N];
    W [N,V,V]; w_r [N,V]; H0 [B,N,K,V] or None (zero state).
    Returns y [B,T,N,V] and H_T [B,N,K,V]; with ``return_states`` also every
    H_t as [B,T,N,K,V] (small problems only).
    """
    v = np.asarray(v, np.float64)
    a = np.asarray(a, np.float64)
    W = np.asarray(W, np.float64)
    w_r = np.asarray(w_r, np.float64)
    B, T, N, V = v.shape
    K = np.shape(q)[-1]
    # Multi-value sharing (Sec. 2.4, N_q = N_k = 1): one q_t, k_t for every head.
    q = np.broadcast_to(np.asarray(q, np.float64), (B, T, N, K))
    k = np.broadcast_to(np.asarray(k, np.float64), (B, T, N, K))
    assert a.shape == (B, T, N)
    assert W.shape == (N, V, V) and w_r.shape == (N, V)

    H = np.zeros((B, N, K, V)) if H0 is None else np.array(H0, dtype=np.float64)
    f = forget_gate(a, alpha, beta)                      # [B,T,N]; input-only (Sec. 2.2)
    y = np.empty((B, T, N, V))
    states = np.empty((B, T, N, K, V)) if return_states else None
    for t in range(T):
        kv = k[:, t, :, :, None] * v[:, t, :, None, :]   # k_t v_t^T   [B,N,K,V]
        Z = np.tanh(np.matmul(H, W) + kv)                # Eq. (10); W broadcast over B
        ft = f[:, t, :, None, None]
        H = ft * H + (1.0 - ft) * Z                      # Eq. (11)
        # Eq. (12): y_t = H_t^T q_t + w_r ⊙ v_t   (sum over the K rows)
        y[:, t] = np.einsum("bnkv,bnk->bnv", H, q[:, t]) + w_r[None] * v[:, t]
        if return_states:
            states[:, t] = H
    if return_states:
        return y, H, states
    return y, H


def m2rnn_forward_scalar(q, k, v, a, alpha, beta, W, w_r, H0=None):
    """The same recurrence as nested pure-Python scalar loops (tiny shapes only).

    Written element by element from Eq. (10)-(13) with the math module, so it
    shares no vectorised routine with ``m2rnn_forward``.
    Arguments are nested lists / arrays indexable as in ``m2rnn_forward``.
    """
    B, T, N, V = len(v), len(v[0]), len(v[0][0]), len(v[0][0][0])
    K = len(q[0][0][0])
    shared = len(q[0][0]) == 1 and N > 1  # one q_t, k_t for all heads (Sec. 2.4)
    y = [[[[0.0] * V for _ in range(N)] for _ in range(T)] for _ in range(B)]
    HT = [[None] * N for _ in range(B)]
    for b in range(B):
        for n in range(N):
            H = [[(0.0 if H0 is None else float(H0[b][n][i][j])) for j in range(V)]
                 for i in range(K)]
            for t in range(T):
                x = float(a[b][t][n]) + float(beta[n])
                sp = math.log1p(math.exp(x)) if x < 30.0 else x + math.log1p(math.exp(-x))
                f = math.exp(-float(alpha[n]) * sp)
                newH = [[0.0] * V for _ in range(K)]
                for i in range(K):
                    for j in range(V):
                        acc = 0.0
                        for l in range(V):
                            acc += H[i][l] * float(W[n][l][j])
                        acc += float(k[b][t][0 if shared else n][i]) * float(v[b][t][n][j])
                        newH[i][j] = f * H[i][j] + (1.0 - f) * math.tanh(acc)
                H = newH
                for j in range(V):
                    s = 0.0
                    for i in range(K):
                        s += H[i][j] * float(q[b][t][0 if shared else n][i])
                    y[b][t][n][j] = s + float(w_r[n][j]) * float(v[b][t][n][j])
            HT[b][n] = H
    return np.array(y, dtype=np.float64), np.array(HT, dtype=np.float64)


def m2rnn_forward_inputs(inp: dict, **kw):
    """``m2rnn_forward`` on a dict of fp64 arrays keyed like the input generator's."""
    return m2rnn_forward(inp["q"], inp["k"], inp["v"], inp["a"], inp["alpha"], inp["beta"],
                         inp["W"], inp["w_r"], inp.get("H0"), **kw)
