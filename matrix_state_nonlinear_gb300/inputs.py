"""Seeded synthetic inputs for the M²RNN forward recurrence.

This module only draws random numbers in the shapes and distributions of the
workloads; it contains none of the recurrence's arithmetic.  Both the CUDA path
(tests, bench) and the fp64 oracle receive the very tensors it returns, so both
sides of a parity comparison see identical bits.

The distributions are this library's synthetic workload recipe:
  q, k ~ N(0, 1/K) (variance 1/K),  v ~ N(0, 1),  gate logits a ~ N(0, 1),
  alpha_n ~ LogUniform[lo, hi] = exp(U[ln lo, ln hi]),  beta_n ~ U[-2, 2],
  W_n = I + N(0, 0.1/V) (variance 0.1/V), optionally rescaled in fp64 to
  spectral norm <= 1 before the cast to the operand dtype,
  w_r ~ N(0, 1),  H0 = 0 or U[-0.5, 0.5].
Shapes and roles follow the symbol table of the M²RNN study notes ("M²RNN:
矩阵状态非线性 RNN 的容量、表达力与系统代价", Sec. 2.1); the identity-centred W
follows their remark that W is initialised to the identity (Sec. 2.3), and
alpha_n > 0 keeps the gate in [0, 1] (Sec. 2.2).

Generation order is fixed: alpha, beta, W, w_r, H0 (from a NumPy PCG64 stream),
then q, k, v, a (from a torch generator on the target device, one seed per
tensor).  The same seed and device give the same bits on every call.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    N: int
    K: int
    V: int
    dtype: str = "bf16"            # operand dtype of q, k, v, a, W: "bf16" or "f32"
    alpha_range: tuple = (0.5, 2.0)
    h0: str = "zero"               # "zero" or "uniform" (U[-0.5, 0.5])
    rescale_w: bool = True         # spectral-norm rescale of W (bf16 workloads)
    shared_qk: bool = False        # one q, k set for all heads: q, k are [B, T, 1, K]

    @property
    def units(self) -> int:
        """Token-head units B*T*N processed by one forward pass."""
        return self.B * self.T * self.N

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads the measurements and parity tests are built around.
WORKLOADS = {
    "tiny_f32_b1_t64_n2_k8_v8": Workload("tiny_f32_b1_t64_n2_k8_v8", 1, 64, 2, 8, 8,
                                         dtype="f32", rescale_w=False),
    "b4_t2048_n8_k64_v64": Workload("b4_t2048_n8_k64_v64", 4, 2048, 8, 64, 64),
    "b8_t16384_n16_k64_v64": Workload("b8_t16384_n16_k64_v64", 8, 16384, 16, 64, 64),
    "b1_t65536_n16_k64_v128": Workload("b1_t65536_n16_k64_v128", 1, 65536, 16, 64, 128),
    "b16_t8192_n32_k128_v128": Workload("b16_t8192_n32_k128_v128", 16, 8192, 32, 128, 128,
                                        alpha_range=(0.1, 4.0), h0="uniform"),
}
WORKLOAD_ORDER = list(WORKLOADS)
# 16K-context training shape: the workload the headline throughput is quoted on.
HEADLINE = "b8_t16384_n16_k64_v64"


def _torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def _spectral_rescale(Wn: np.ndarray) -> np.ndarray:
    """Scale one V x V matrix down so its largest singular value is <= 1."""
    s = np.linalg.svd(Wn, compute_uv=False)[0]
    return Wn / max(1.0, float(s))


def make_params(wl: Workload, seed: int = 0) -> dict:
    """Per-head parameters and the initial state, drawn on the CPU in fp64.

    Returns fp64 NumPy arrays before any cast (alpha, beta [N]; W [N,V,V];
    w_r [N,V]; H0 [B,N,K,V] or None).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    lo, hi = wl.alpha_range
    alpha = np.exp(rng.uniform(math.log(lo), math.log(hi), size=wl.N))
    beta = rng.uniform(-2.0, 2.0, size=wl.N)
    W = np.eye(wl.V)[None] + rng.normal(0.0, math.sqrt(0.1 / wl.V), size=(wl.N, wl.V, wl.V))
    if wl.rescale_w:
        W = np.stack([_spectral_rescale(W[n]) for n in range(wl.N)])
    w_r = rng.normal(0.0, 1.0, size=(wl.N, wl.V))
    if wl.h0 == "uniform":
        H0 = rng.uniform(-0.5, 0.5, size=(wl.B, wl.N, wl.K, wl.V))
    else:
        H0 = None
    return dict(alpha=alpha, beta=beta, W=W, w_r=w_r, H0=H0)


def _randn(shape, std, seed, device, dtype):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def make_inputs(wl: Workload, device="cpu", seed: int = 0) -> dict:
    """All inputs of one forward pass as torch tensors on ``device``.

    q, k [B,T,N,K] (or [B,T,1,K] when shared_qk); v [B,T,N,V]; a [B,T,N]; W [N,V,V]
    in the operand dtype;
    alpha, beta [N]; w_r [N,V]; H0 [B,N,K,V] (or None) in float32.
    All tensors are contiguous.
    """
    dev = torch.device(device)
    p = make_params(wl, seed)
    dt = _torch_dtype(wl.dtype)
    out = dict(
        alpha=torch.tensor(p["alpha"], dtype=torch.float32, device=dev),
        beta=torch.tensor(p["beta"], dtype=torch.float32, device=dev),
        W=torch.tensor(p["W"], dtype=torch.float32).to(dt).to(dev).contiguous(),
        w_r=torch.tensor(p["w_r"], dtype=torch.float32, device=dev),
        H0=None if p["H0"] is None else torch.tensor(p["H0"], dtype=torch.float32, device=dev),
    )
    B, T, N, K, V = wl.B, wl.T, wl.N, wl.K, wl.V
    base = seed * 1000 + 17
    Nqk = 1 if wl.shared_qk else N
    out["q"] = _randn((B, T, Nqk, K), 1.0 / math.sqrt(K), base + 0, dev, dt)
    out["k"] = _randn((B, T, Nqk, K), 1.0 / math.sqrt(K), base + 1, dev, dt)
    out["v"] = _randn((B, T, N, V), 1.0, base + 2, dev, dt)
    out["a"] = _randn((B, T, N), 1.0, base + 3, dev, dt)
    return out


def to_f64_numpy(t: torch.Tensor | None) -> np.ndarray | None:
    """Exact upcast of a (bf16 or f32) tensor to an fp64 NumPy array on the host."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()


def slice_pair(inp: dict, b: int, n: int) -> dict:
    """The inputs of one (batch, head) pair as a B=1, N=1 problem (fp64 host arrays).

    Pairs are independent units of the recurrence, so an oracle run on this
    slice gives exactly that pair's outputs of the full problem.
    """
    s = {}
    for key in ("v", "a"):
        s[key] = to_f64_numpy(inp[key][b:b + 1, :, n:n + 1])
    for key in ("q", "k"):  # a shared q, k (one head) serves every head
        h = n if inp[key].shape[2] > 1 else 0
        s[key] = to_f64_numpy(inp[key][b:b + 1, :, h:h + 1])
    s["alpha"] = to_f64_numpy(inp["alpha"][n:n + 1])
    s["beta"] = to_f64_numpy(inp["beta"][n:n + 1])
    s["W"] = to_f64_numpy(inp["W"][n:n + 1])
    s["w_r"] = to_f64_numpy(inp["w_r"][n:n + 1])
    s["H0"] = None if inp["H0"] is None else to_f64_numpy(inp["H0"][b:b + 1, n:n + 1])
    return s


def all_f64(inp: dict) -> dict:
    """Every input as an fp64 host array (small problems only)."""
    return {key: to_f64_numpy(val) for key, val in inp.items()}
