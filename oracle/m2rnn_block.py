"""fp64 CPU oracle for the M²RNN block's prologue and epilogue.  TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The CUDA library never calls it and shares
no code with it.

Source: the M²RNN study notes ("M²RNN: 矩阵状态非线性 RNN 的容量、表达力与系统代价"),
Sec. 2.3 (the paper's Eq. (14)-(23), Fig. 2):
  * q, k, v each go through a linear projection, a depthwise causal Conv1D of
    kernel size 4, and SiLU; the convolution reads only the current and earlier
    positions;
  * the output gate g_t = SiLU(W_g x_t) has no convolution;
  * after the recurrence: y_gt = RMSNorm(y_t ⊙ g_t) (gate first, then the norm),
    then W_o back to the model width.
Appendix C (notes, "RMSNormTP"): the norm's statistic is one scalar per token over
the whole width, s = [ (1/d) sum_j x_j^2 ]^(-1/2), with a learnable weight w_i;
the notes add that the paper leaves out the stabilising epsilon for brevity.

Readings taken where the notes leave a step open:
  * Conv1D: out[t, c] = sum_{j=0..3} w[c, j] * x[t - 3 + j, c] (+ bias[c]), with
    x at negative times equal to zero (causal, left zero padding); the bias is
    optional (absent unless given).
  * SiLU(x) = x * sigmoid(x).
  * RMSNorm over the d = N * V values of one token (all heads, as the tensor-
    parallel statistic of Appendix C implies), out_i = w_i x_i / sqrt(mean(x^2) + eps).
  * The projections W_q, W_k, W_v, W_g, W_f, W_o are plain matrix products outside
    these functions.
"""
from __future__ import annotations

import numpy as np

KERNEL = 4  # Conv1D kernel size (Sec. 2.3)


def silu(x):
    """x * sigmoid(x), overflow-free."""
    x = np.asarray(x, np.float64)
    e = np.exp(-np.abs(x))
    sig = np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))
    return x * sig


def causal_conv1d(x, w, bias=None):
    """Depthwise causal Conv1D over time: x [B, T, C], w [C, KERNEL], bias [C] or None."""
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    B, T, C = x.shape
    out = np.zeros((B, T, C))
    for j in range(KERNEL):
        shift = KERNEL - 1 - j          # tap j reads x[t - shift]
        if shift >= T:
            continue
        out[:, shift:, :] += w[None, None, :, j] * x[:, :T - shift, :]
    if bias is not None:
        out += np.asarray(bias, np.float64)[None, None, :]
    return out


def conv_silu(x, w, bias=None):
    """The q / k / v prologue: SiLU(causal depthwise Conv1D(x))."""
    return silu(causal_conv1d(x, w, bias))


def gate_rmsnorm(y, g_pre, w_norm, eps):
    """The epilogue: RMSNorm(y ⊙ SiLU(g_pre)) over the last axis (d = N * V per token)."""
    z = np.asarray(y, np.float64) * silu(g_pre)
    ms = np.mean(z * z, axis=-1, keepdims=True)
    return np.asarray(w_norm, np.float64) * z / np.sqrt(ms + eps)
