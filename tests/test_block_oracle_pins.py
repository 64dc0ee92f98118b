"""Pins for the block prologue / epilogue oracle (the M²RNN notes' Sec. 2.3 and
Appendix C), each against a library routine, a closed form or an invariant:
  * causal depthwise Conv1D == torch.nn.functional.conv1d (groups = C, left
    padding 3) in fp64; causality: output at t never changes when later inputs do;
  * SiLU: x * expit(x) (scipy), SiLU(x) - SiLU(-x) = x, SiLU(0) = 0;
  * RMSNorm == torch.nn.functional.rms_norm in fp64 on y ⊙ SiLU(g);
  * gate before norm: with eps = 0 the output does not change when the gate
    activation is scaled by a constant (a norm applied before the gate would);
  * the statistic spans the whole token: changing one head changes every head's
    output.
A mutation test plants mistakes in a copy and checks a pin fails for each.
"""
import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

from oracle.m2rnn_block import KERNEL, causal_conv1d, conv_silu, gate_rmsnorm, silu


def conv_ref_torch(x, w, bias):
    xt = torch.from_numpy(np.ascontiguousarray(np.moveaxis(x, 1, 2)))           # [B, C, T]
    wt = torch.from_numpy(np.asarray(w)[:, None, :])                              # [C, 1, 4]
    bt = None if bias is None else torch.from_numpy(np.asarray(bias))
    out = F.conv1d(F.pad(xt, (KERNEL - 1, 0)), wt, bt, groups=x.shape[2])
    return np.moveaxis(out.numpy(), 1, 2)


def pin_conv_matches_torch(conv):
    rng = np.random.default_rng(1)
    for (B, T, C) in [(2, 9, 5), (1, 2, 3), (3, 40, 8)]:
        x = rng.normal(size=(B, T, C))
        w = rng.normal(size=(C, KERNEL))
        b = rng.normal(size=C)
        for bias in (None, b):
            if not np.allclose(conv(x, w, bias), conv_ref_torch(x, w, bias), rtol=1e-13, atol=1e-13):
                return False
    return True


def pin_conv_causal(conv):
    rng = np.random.default_rng(2)
    x = rng.normal(size=(2, 30, 4))
    w = rng.normal(size=(4, KERNEL))
    base = conv(x, w, None)
    x2 = x.copy()
    x2[:, 17:] = rng.normal(size=x2[:, 17:].shape)
    return np.array_equal(conv(x2, w, None)[:, :17], base[:, :17])


def pin_silu(silu_fn):
    x = np.linspace(-40, 40, 801)
    return (np.allclose(silu_fn(x), x * scipy.special.expit(x), rtol=1e-14, atol=1e-300)
            and np.allclose(silu_fn(x) - silu_fn(-x), x, atol=1e-12) and silu_fn(np.array(0.0)) == 0)


def pin_rmsnorm_matches_torch(gr):
    rng = np.random.default_rng(3)
    y = rng.normal(size=(3, 5, 48))
    g = rng.normal(size=(3, 5, 48))
    w = rng.normal(size=48)
    for eps in (0.0, 1e-6, 0.5):
        z = torch.from_numpy(y * (g * scipy.special.expit(g)))
        ref = F.rms_norm(z, (48,), torch.from_numpy(w), eps=eps).numpy()
        if not np.allclose(gr(y, g, w, eps), ref, rtol=1e-12, atol=1e-12):
            return False
    return True


def pin_gate_before_norm(gr):
    """eps = 0: scaling y's gate by c > 0 (via y -> c y) leaves the output unchanged,
    and so does scaling the gated product; a norm taken before gating would carry
    the gate's scale into the output."""
    rng = np.random.default_rng(4)
    y = rng.normal(size=(2, 3, 32))
    g = rng.normal(size=(2, 3, 32)) + 3.0          # SiLU(g) ~ g: far from zero
    w = rng.normal(size=32)
    out = gr(y, g, w, 0.0)
    return np.allclose(gr(2.5 * y, g, w, 0.0), out, rtol=1e-12) and not np.allclose(
        gr(y, g + 1.0, w, 0.0), out, rtol=1e-3)


def pin_stat_spans_token(gr):
    rng = np.random.default_rng(5)
    y = rng.normal(size=(1, 1, 64))
    g = rng.normal(size=(1, 1, 64))
    w = np.ones(64)
    y2 = y.copy()
    y2[..., 48:] *= 3.0                            # change only the last "head"
    a, b = gr(y, g, w, 1e-6), gr(y2, g, w, 1e-6)
    return not np.allclose(a[..., :48], b[..., :48], rtol=1e-6)


CONV_PINS = [pin_conv_matches_torch, pin_conv_causal]
NORM_PINS = [pin_rmsnorm_matches_torch, pin_gate_before_norm, pin_stat_spans_token]


@pytest.mark.parametrize("pin", CONV_PINS, ids=lambda f: f.__name__)
def test_conv_pin(pin):
    assert pin(causal_conv1d)


def test_silu_pin():
    assert pin_silu(silu)


@pytest.mark.parametrize("pin", NORM_PINS, ids=lambda f: f.__name__)
def test_norm_pin(pin):
    assert pin(gate_rmsnorm)


def test_conv_silu_composes():
    rng = np.random.default_rng(6)
    x = rng.normal(size=(2, 7, 3))
    w = rng.normal(size=(3, KERNEL))
    assert np.array_equal(conv_silu(x, w), silu(causal_conv1d(x, w)))


# ---------------------------------------------------------------- mutation test
def conv_mutant(kind):
    def conv(x, w, bias=None):
        B, T, C = x.shape
        out = np.zeros((B, T, C))
        for j in range(KERNEL):
            shift = KERNEL - 1 - j
            if kind == "taps_reversed":
                shift = j
            if kind == "acausal" and j == KERNEL - 1:
                out[:, :T - 1] += w[None, None, :, j] * x[:, 1:]
                continue
            if shift >= T:
                continue
            out[:, shift:, :] += w[None, None, :, j] * x[:, :T - shift, :]
        if bias is not None and kind != "bias_dropped":
            out += bias[None, None, :]
        return out
    return conv


def norm_mutant(kind):
    def gr(y, g, w, eps):
        if kind == "norm_then_gate":
            ms = np.mean(y * y, axis=-1, keepdims=True)
            return w * y / np.sqrt(ms + eps) * silu(g)
        z = y * (silu(g) if kind != "sigmoid_gate" else scipy.special.expit(g))
        if kind == "per_head_stat":
            zz = z.reshape(*z.shape[:-1], -1, 16)
            ms = np.mean(zz * zz, axis=-1, keepdims=True)
            return w * (zz / np.sqrt(ms + eps)).reshape(z.shape)
        ms = np.mean(z * z, axis=-1, keepdims=True)
        if kind == "eps_outside":
            return w * z / (np.sqrt(ms) + eps)
        return w * z / np.sqrt(ms + eps)
    return gr


@pytest.mark.parametrize("kind", ["taps_reversed", "acausal", "bias_dropped"])
def test_conv_mutant_fails_a_pin(kind):
    assert not all(p(conv_mutant(kind)) for p in CONV_PINS)


@pytest.mark.parametrize("kind", ["norm_then_gate", "sigmoid_gate", "per_head_stat", "eps_outside"])
def test_norm_mutant_fails_a_pin(kind):
    assert not all(p(norm_mutant(kind)) for p in NORM_PINS)


def test_unmutated_copies_pass():
    assert all(p(conv_mutant("none")) for p in CONV_PINS)
    assert all(p(norm_mutant("none")) for p in NORM_PINS)
