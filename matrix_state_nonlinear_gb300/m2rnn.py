"""Thin Python binding of the C ABI in include/m2rnn.h (argument marshalling only).

Every step of the recurrence runs in the CUDA kernels of libm2rnn.so; this
module checks tensor dtypes, devices and contiguity, passes raw device pointers
and the current CUDA stream, and turns status codes into exceptions.  There is
no CPU fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libm2rnn.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4

# Exported symbols of include/m2rnn.h, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
SYMBOLS = {
    "m2rnn_forward_f32": (_I, [_P] * 11 + [_I] * 5 + [_P]),
    "m2rnn_forward_bf16": (_I, [_P] * 11 + [_I] * 5 + [_P]),
    "m2rnn_forward_bf16_variant": (_I, [_P] * 11 + [_I] * 6 + [_P]),
    "m2rnn_forward_f32_qk": (_I, [_P] * 11 + [_I] * 6 + [_P]),
    "m2rnn_forward_bf16_qk": (_I, [_P] * 11 + [_I] * 7 + [_P]),
    "m2rnn_variant_name": (ctypes.c_char_p, [_I]),
    "m2rnn_pick_variant": (_I, [_I] * 5),
    "m2rnn_variant_supports": (_I, [_I] * 6),
    "m2rnn_balanced_stretch": (_I, [ctypes.c_longlong, _I, ctypes.c_longlong, ctypes.c_longlong,
                                    ctypes.POINTER(ctypes.c_longlong),
                                    ctypes.POINTER(ctypes.c_longlong)]),
    "m2rnn_stream_status": (_I, [_P]),
    "m2rnn_status_string": (ctypes.c_char_p, [_I]),
    "m2rnn_version": (_I, []),
    "m2rnn_forward_train_f32": (_I, [_P] * 12 + [_I] * 6 + [_P]),
    "m2rnn_forward_train_bf16": (_I, [_P] * 12 + [_I] * 6 + [_P]),
    "m2rnn_backward_workspace_bytes": (ctypes.c_size_t, [_I] * 6),
    "m2rnn_backward_f32": (_I, [_P] * 21 + [_I] * 6 + [_P, ctypes.c_size_t, _P]),
    "m2rnn_backward_bf16": (_I, [_P] * 21 + [_I] * 7 + [_P, ctypes.c_size_t, _P]),
    "m2rnn_backward_bf16_noalloc": (_I, [_P] * 21 + [_I] * 6 + [_P]),
    "m2rnn_decode_step_bf16": (_I, [_P] * 11 + [_I] * 5 + [_P]),
    "m2rnn_decode_step_bf16_variant": (_I, [_P] * 11 + [_I] * 6 + [_P]),
    "m2rnn_conv_silu_bf16": (_I, [_P] * 4 + [_I] * 3 + [_P]),
    "m2rnn_forward_conv_bf16": (_I, [_P] * 17 + [_I] * 6 + [_P]),
    "m2rnn_gate_rmsnorm_bf16": (_I, [_P] * 3 + [ctypes.c_float, _P, ctypes.c_longlong, _I, _P]),
}

_lib = None


class M2RNNError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status) if _lib else status} (status {status})")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libm2rnn.so once; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libm2rnn.so not found at {path}; build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SYMBOLS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().m2rnn_status_string(int(status)).decode()


def version() -> int:
    return load_library().m2rnn_version()


def variant_name(variant: int) -> str | None:
    s = load_library().m2rnn_variant_name(int(variant))
    return None if s is None else s.decode()


def pick_variant(B: int, T: int, N: int, K: int, V: int) -> int:
    return load_library().m2rnn_pick_variant(B, T, N, K, V)


def variant_supports(variant: int, B: int, T: int, N: int, K: int, V: int) -> bool:
    return bool(load_library().m2rnn_variant_supports(variant, B, T, N, K, V))


def balanced_stretch(pairs: int, T: int, workers: int, worker: int) -> tuple[int, int]:
    """Positions [begin, end) of the steps line that block `worker` of the balanced K = V = 128
    forward runs (pair p owns [p T, (p + 1) T))."""
    b, e = ctypes.c_longlong(), ctypes.c_longlong()
    st = load_library().m2rnn_balanced_stretch(pairs, T, workers, worker, ctypes.byref(b),
                                               ctypes.byref(e))
    if st != 0:
        raise ValueError(f"invalid balanced schedule arguments {pairs, T, workers, worker}")
    return b.value, e.value


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def stream_status(stream=None) -> int:
    """Synchronises the stream; returns (and clears) the device status (OK or ERR_TIMEOUT)."""
    return load_library().m2rnn_stream_status(ctypes.c_void_p(_stream_ptr(stream)))


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _check(t, name, dtype, shape, dev):
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device != dev:
        raise ValueError(f"{name}: expected device {dev}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def _marshal(q, k, v, a, alpha, beta, W, w_r, H0, y, H_T, opdtype):
    """Checks tensors and returns (pointers, (B, T, N, K, V), y, Nqk).

    q and k may have N heads or a single head shared by all heads of v.
    """
    if q.device.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, T, Nqk, K = q.shape
    N, V = v.shape[2], v.shape[3]
    dev = q.device
    if Nqk not in (1, N):
        raise ValueError(f"q, k must have 1 or {N} heads, got {Nqk}")
    for t, name, dt, shp in [(q, "q", opdtype, (B, T, Nqk, K)), (k, "k", opdtype, (B, T, Nqk, K)),
                             (v, "v", opdtype, (B, T, N, V)), (a, "a", opdtype, (B, T, N)),
                             (alpha, "alpha", torch.float32, (N,)),
                             (beta, "beta", torch.float32, (N,)),
                             (W, "W", opdtype, (N, V, V)), (w_r, "w_r", torch.float32, (N, V)),
                             (H0, "H0", torch.float32, (B, N, K, V))]:
        _check(t, name, dt, shp, dev)
    if y is None:
        y = torch.empty((B, T, N, V), dtype=torch.float32, device=dev)
    _check(y, "y", torch.float32, (B, T, N, V), dev)
    if H_T is not None:
        _check(H_T, "H_T", torch.float32, (B, N, K, V), dev)
    ptrs = [_ptr(x) for x in (q, k, v, a, alpha, beta, W, w_r, H0, y, H_T)]
    return ptrs, (B, T, N, K, V), y, Nqk


def m2rnn_forward_f32(q, k, v, a, alpha, beta, W, w_r, H0=None, y=None, H_T=None, stream=None):
    """fp32-operand forward (all tensors float32).  Returns (y, H_T)."""
    lib = load_library()
    ptrs, (B, T, N, K, V), y, Nqk = _marshal(q, k, v, a, alpha, beta, W, w_r, H0, y, H_T,
                                              torch.float32)
    if Nqk == N:
        st = lib.m2rnn_forward_f32(*ptrs, B, T, N, K, V, ctypes.c_void_p(_stream_ptr(stream)))
    else:
        st = lib.m2rnn_forward_f32_qk(*ptrs, B, T, N, Nqk, K, V,
                                      ctypes.c_void_p(_stream_ptr(stream)))
    if st != OK:
        raise M2RNNError(st, "m2rnn_forward_f32")
    return y, H_T


def m2rnn_forward_bf16_variant(q, k, v, a, alpha, beta, W, w_r, H0=None, y=None, H_T=None,
                               variant=0, stream=None):
    """bf16-operand / fp32-state forward with an explicit kernel variant (0 = auto)."""
    lib = load_library()
    ptrs, (B, T, N, K, V), y, Nqk = _marshal(q, k, v, a, alpha, beta, W, w_r, H0, y, H_T,
                                              torch.bfloat16)
    if Nqk == N:
        st = lib.m2rnn_forward_bf16_variant(*ptrs, B, T, N, K, V, int(variant),
                                            ctypes.c_void_p(_stream_ptr(stream)))
    else:
        st = lib.m2rnn_forward_bf16_qk(*ptrs, B, T, N, Nqk, K, V, int(variant),
                                       ctypes.c_void_p(_stream_ptr(stream)))
    if st != OK:
        raise M2RNNError(st, "m2rnn_forward_bf16")
    return y, H_T


def m2rnn_forward_bf16(q, k, v, a, alpha, beta, W, w_r, H0=None, y=None, H_T=None, stream=None):
    """bf16-operand / fp32-state forward (q, k, v, a, W bfloat16; the rest float32)."""
    lib = load_library()
    ptrs, (B, T, N, K, V), y, Nqk = _marshal(q, k, v, a, alpha, beta, W, w_r, H0, y, H_T,
                                              torch.bfloat16)
    if Nqk != N:
        return m2rnn_forward_bf16_variant(q, k, v, a, alpha, beta, W, w_r, H0, y, H_T, 0, stream)
    st = lib.m2rnn_forward_bf16(*ptrs, B, T, N, K, V, ctypes.c_void_p(_stream_ptr(stream)))
    if st != OK:
        raise M2RNNError(st, "m2rnn_forward_bf16")
    return y, H_T


def m2rnn_forward(inputs: dict, y=None, H_T=None, variant=0, stream=None):
    """Forward pass on a dict keyed like the input generator's output.

    Dispatches on the operand dtype of q: float32 -> the fp32 path, bfloat16 ->
    the tensor-core path.  q and k with a single head are shared by all heads.
    Allocates y and H_T (torch memory) when not given.
    """
    q = inputs["q"]
    B, T, _, K = q.shape
    N, V = inputs["v"].shape[2], inputs["v"].shape[3]
    if H_T is None:
        H_T = torch.empty((B, N, K, V), dtype=torch.float32, device=q.device)
    args = [inputs[x] for x in ("q", "k", "v", "a", "alpha", "beta", "W", "w_r")]
    if q.dtype == torch.float32:
        return m2rnn_forward_f32(*args, inputs.get("H0"), y, H_T, stream=stream)
    return m2rnn_forward_bf16_variant(*args, inputs.get("H0"), y, H_T, variant=variant,
                                      stream=stream)


def m2rnn_forward_conv(inputs: dict, conv: dict, y=None, H_T=None, stream=None):
    """The block prologue fused into the bf16 forward: inputs["q"], ["k"], ["v"] are the raw
    projections (bf16, shaped like q, k, v); conv holds the causal conv's taps "wq", "wk", "wv"
    ([C, 4] float32, C = heads x width) and biases "bq", "bk", "bv" ([C] float32 or None).
    Returns (y, H_T), the bits of conv_silu on each projection followed by m2rnn_forward."""
    lib = load_library()
    args = [inputs[x] for x in ("q", "k", "v", "a", "alpha", "beta", "W", "w_r")]
    ptrs, (B, T, N, K, V), y, Nqk = _marshal(*args, inputs.get("H0"), y, H_T, torch.bfloat16)
    if H_T is None:
        H_T = torch.empty((B, N, K, V), dtype=torch.float32, device=y.device)
        ptrs[10] = _ptr(H_T)
    dev = y.device
    taps = []
    for name, C in (("q", Nqk * K), ("k", Nqk * K), ("v", N * V)):
        w, b = conv["w" + name], conv.get("b" + name)
        _check(w, "w" + name, torch.float32, (C, 4), dev)
        _check(b, "b" + name, torch.float32, (C,), dev)
        taps += [_ptr(w), _ptr(b)]
    st = lib.m2rnn_forward_conv_bf16(*ptrs[:3], *taps, *ptrs[3:], B, T, N, Nqk, K, V,
                                     ctypes.c_void_p(_stream_ptr(stream)))
    if st != OK:
        raise M2RNNError(st, "m2rnn_forward_conv_bf16")
    return y, H_T


# ---------------------------------------------------------------- training support
def _shape_of(inputs):
    q, v = inputs["q"], inputs["v"]
    B, T, Nqk, K = q.shape
    return B, T, v.shape[2], Nqk, K, v.shape[3]


def m2rnn_forward_train(inputs: dict, y=None, H_T=None, Hs=None, stream=None):
    """Forward pass that also keeps every step's state for the backward pass.

    Returns (y, H_T, Hs) with Hs [B, N, T, K, V] (Hs[:, :, t] = H_t): float32 on the
    fp32 path, bfloat16 (the rounding the tensor cores consume) on the bf16 path.
    Dispatches on the operand dtype of q like ``m2rnn_forward``.
    """
    lib = load_library()
    B, T, N, Nqk, K, V = _shape_of(inputs)
    q = inputs["q"]
    dev = q.device
    if H_T is None:
        H_T = torch.empty((B, N, K, V), dtype=torch.float32, device=dev)
    opdtype = torch.float32 if q.dtype == torch.float32 else torch.bfloat16
    if Hs is None:
        Hs = torch.empty((B, N, T, K, V), dtype=opdtype, device=dev)
    _check(Hs, "Hs", opdtype, (B, N, T, K, V), dev)
    args = [inputs[x] for x in ("q", "k", "v", "a", "alpha", "beta", "W", "w_r")]
    ptrs, _, y, _ = _marshal(*args, inputs.get("H0"), y, H_T, opdtype)
    fn = lib.m2rnn_forward_train_f32 if opdtype == torch.float32 else lib.m2rnn_forward_train_bf16
    st = fn(*ptrs, _ptr(Hs), B, T, N, Nqk, K, V, ctypes.c_void_p(_stream_ptr(stream)))
    if st != OK:
        raise M2RNNError(st, "m2rnn_forward_train")
    return y, H_T, Hs


def backward_workspace_bytes(B, T, N, Nqk, K, V) -> int:
    return int(load_library().m2rnn_backward_workspace_bytes(B, T, N, Nqk, K, V))


def m2rnn_backward(inputs: dict, Hs, dy, dH_T=None, grads=None, workspace=None, variant=0,
                   stream=None):
    """Backward pass: gradients of a loss through y (dy) and H_T (dH_T, optional).

    ``Hs`` is the state history from ``m2rnn_forward_train`` on the same inputs.
    Returns a dict dq, dk, dv, da, dalpha, dbeta, dW, dw_r, dH0 (float32; ``grads``
    may supply any of them preallocated).  The workspace is allocated (torch
    memory) when not given.
    """
    lib = load_library()
    B, T, N, Nqk, K, V = _shape_of(inputs)
    q = inputs["q"]
    dev = q.device
    opdtype = torch.float32 if q.dtype == torch.float32 else torch.bfloat16
    args = [inputs[x] for x in ("q", "k", "v", "a", "alpha", "beta", "W", "w_r")]
    ptrs, _, _, _ = _marshal(*args, inputs.get("H0"), dy, None, opdtype)
    _check(Hs, "Hs", opdtype, (B, N, T, K, V), dev)
    _check(dy, "dy", torch.float32, (B, T, N, V), dev)
    _check(dH_T, "dH_T", torch.float32, (B, N, K, V), dev)
    shapes = {"dq": (B, T, Nqk, K), "dk": (B, T, Nqk, K), "dv": (B, T, N, V), "da": (B, T, N),
              "dalpha": (N,), "dbeta": (N,), "dW": (N, V, V), "dw_r": (N, V),
              "dH0": (B, N, K, V)}
    out = dict(grads or {})
    for name, shp in shapes.items():
        if name not in out:
            out[name] = torch.empty(shp, dtype=torch.float32, device=dev)
        _check(out[name], name, torch.float32, shp, dev)
    nbytes = backward_workspace_bytes(B, T, N, Nqk, K, V)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    gptrs = [_ptr(out[n]) for n in shapes]
    common = ptrs[:9] + [_ptr(Hs), _ptr(dy), _ptr(dH_T)] + gptrs
    sp = ctypes.c_void_p(_stream_ptr(stream))
    if opdtype == torch.float32:
        st = lib.m2rnn_backward_f32(*common, B, T, N, Nqk, K, V, _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), sp)
    else:
        st = lib.m2rnn_backward_bf16(*common, B, T, N, Nqk, K, V, int(variant), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), sp)
    if st != OK:
        raise M2RNNError(st, "m2rnn_backward")
    return out


def m2rnn_backward_noalloc(inputs: dict, Hs, dy, dH_T=None, grads=None, stream=None):
    """``m2rnn_backward`` on bf16 inputs with the library's own fixed scratch instead of a
    workspace (at most 16 MiB of workspace; calls on one device must not overlap)."""
    lib = load_library()
    B, T, N, Nqk, K, V = _shape_of(inputs)
    q = inputs["q"]
    dev = q.device
    args = [inputs[x] for x in ("q", "k", "v", "a", "alpha", "beta", "W", "w_r")]
    ptrs, _, _, _ = _marshal(*args, inputs.get("H0"), dy, None, torch.bfloat16)
    _check(Hs, "Hs", torch.bfloat16, (B, N, T, K, V), dev)
    _check(dH_T, "dH_T", torch.float32, (B, N, K, V), dev)
    shapes = {"dq": (B, T, Nqk, K), "dk": (B, T, Nqk, K), "dv": (B, T, N, V), "da": (B, T, N),
              "dalpha": (N,), "dbeta": (N,), "dW": (N, V, V), "dw_r": (N, V),
              "dH0": (B, N, K, V)}
    out = dict(grads or {})
    for name, shp in shapes.items():
        if name not in out:
            out[name] = torch.empty(shp, dtype=torch.float32, device=dev)
        _check(out[name], name, torch.float32, shp, dev)
    st = lib.m2rnn_backward_bf16_noalloc(*ptrs[:9], _ptr(Hs), _ptr(dy), _ptr(dH_T),
                                         *[_ptr(out[n]) for n in shapes], B, T, N, Nqk, K, V,
                                         ctypes.c_void_p(_stream_ptr(stream)))
    if st != OK:
        raise M2RNNError(st, "m2rnn_backward_bf16_noalloc")
    return out


def m2rnn_decode_step(q, k, v, a, alpha, beta, W, w_r, H_in, H_out=None, y=None, stream=None,
                      variant=0):
    """One decode step (bf16 operands): q, k [B, Nqk, K]; v [B, N, V]; a [B, N]; state
    H_in [B, N, K, V] float32 (None: zero).  Writes H_out (defaults to H_in, in place,
    when H_in is given) and y [B, N, V]; returns (y, H_out).  variant: 0 automatic,
    1 one block per pair, 2 the persistent kernel (K = V = 64)."""
    lib = load_library()
    B, Nqk, K = q.shape
    N, V = v.shape[1], v.shape[2]
    dev = q.device
    if q.device.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    for t, name, dt, shp in [(q, "q", torch.bfloat16, (B, Nqk, K)),
                             (k, "k", torch.bfloat16, (B, Nqk, K)),
                             (v, "v", torch.bfloat16, (B, N, V)), (a, "a", torch.bfloat16, (B, N)),
                             (alpha, "alpha", torch.float32, (N,)),
                             (beta, "beta", torch.float32, (N,)),
                             (W, "W", torch.bfloat16, (N, V, V)),
                             (w_r, "w_r", torch.float32, (N, V)),
                             (H_in, "H_in", torch.float32, (B, N, K, V))]:
        _check(t, name, dt, shp, dev)
    if H_out is None:
        H_out = H_in if H_in is not None else torch.empty((B, N, K, V), dtype=torch.float32,
                                                          device=dev)
    _check(H_out, "H_out", torch.float32, (B, N, K, V), dev)
    if y is None:
        y = torch.empty((B, N, V), dtype=torch.float32, device=dev)
    _check(y, "y", torch.float32, (B, N, V), dev)
    ptrs = [_ptr(x) for x in (q, k, v, a, alpha, beta, W, w_r, H_in, H_out, y)]
    if variant == 0:
        st = lib.m2rnn_decode_step_bf16(*ptrs, B, N, Nqk, K, V,
                                        ctypes.c_void_p(_stream_ptr(stream)))
    else:
        st = lib.m2rnn_decode_step_bf16_variant(*ptrs, B, N, Nqk, K, V, int(variant),
                                                ctypes.c_void_p(_stream_ptr(stream)))
    if st != OK:
        raise M2RNNError(st, "m2rnn_decode_step_bf16")
    return y, H_out


# ---------------------------------------------------------------- block prologue / epilogue
def conv_silu(x, w, bias=None, out=None, stream=None):
    """SiLU(causal depthwise Conv1D, kernel 4) over time: x [B, T, C] bf16, w [C, 4] float32,
    bias [C] float32 or None.  Returns out [B, T, C] bf16."""
    lib = load_library()
    if x.device.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, T, C = x.shape
    dev = x.device
    _check(x, "x", torch.bfloat16, (B, T, C), dev)
    _check(w, "w", torch.float32, (C, 4), dev)
    _check(bias, "bias", torch.float32, (C,), dev)
    if out is None:
        out = torch.empty_like(x)
    _check(out, "out", torch.bfloat16, (B, T, C), dev)
    st = lib.m2rnn_conv_silu_bf16(_ptr(x), _ptr(w), _ptr(bias), _ptr(out), B, T, C,
                                  ctypes.c_void_p(_stream_ptr(stream)))
    if st != OK:
        raise M2RNNError(st, "m2rnn_conv_silu_bf16")
    return out


def gate_rmsnorm(y, g_pre, w_norm, eps=1e-6, out=None, stream=None):
    """RMSNorm(y ⊙ SiLU(g_pre)) over the last axis: y [..., D] float32, g_pre [..., D] bf16,
    w_norm [D] float32.  Returns out [..., D] bf16."""
    lib = load_library()
    if y.device.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    D = y.shape[-1]
    rows = y.numel() // D if D else 0
    dev = y.device
    _check(y, "y", torch.float32, tuple(y.shape), dev)
    _check(g_pre, "g_pre", torch.bfloat16, tuple(y.shape), dev)
    _check(w_norm, "w_norm", torch.float32, (D,), dev)
    if out is None:
        out = torch.empty(y.shape, dtype=torch.bfloat16, device=dev)
    _check(out, "out", torch.bfloat16, tuple(y.shape), dev)
    st = lib.m2rnn_gate_rmsnorm_bf16(_ptr(y), _ptr(g_pre), _ptr(w_norm), float(eps), _ptr(out),
                                     rows, D, ctypes.c_void_p(_stream_ptr(stream)))
    if st != OK:
        raise M2RNNError(st, "m2rnn_gate_rmsnorm_bf16")
    return out
