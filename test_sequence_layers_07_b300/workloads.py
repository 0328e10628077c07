"""Seeded synthetic inputs for the TTT inner-loop scan.

This module only draws and rounds random numbers; it holds none of the
method's arithmetic.  The same rounded values feed the CUDA library and the
fp64 oracle used by the tests.

Recipe (all draws from ``numpy.random.default_rng(seed)`` (PCG64), in float64,
in the order listed):

* q, k, v ~ N(0, 1/d) i.i.d., shape [B, H, T, d], drawn in the order Q, K, V.
* rows of K (and of Q unless ``normalize_q`` is False) are scaled to unit L2
  norm; V is never normalised.
* per-token step size eta_t = sigmoid(u_t) / d with u_t ~ N(0, 1), shape
  [B, H, T]; or a constant when ``eta_const`` is given.
* initial fast weights ~ N(0, w_std^2) fp32, one draw per head broadcast over
  the batch (W0 [H, d, d] -> [B, H, d, d]); or zeros.
* for TTT-MLP, W1 [H, d, hd] then W2 [H, hd, d] ~ N(0, w_std^2), broadcast
  over the batch.

Rounding: float64 -> float32 (round to nearest even), then for bf16 inputs
float32 -> bfloat16 (round to nearest even, done by torch on the CPU).  eta and
the weights are always fp32.  The oracle reads exactly these rounded values,
widened to float64.

The named workloads are those the library is measured and checked on:
``oracle_check`` (d=16, fp32), ``linear_prefill`` (B=8, H=12, d=64, T=2048,
b=16, bf16), ``mlp_prefill`` (same tokens, hidden 256), ``long_context``
(B=1, H=16, d=128, T=32768, b in {16, 64, 512}), ``decode`` (B=256, H=12,
d=64, 1024 single-token steps, per-sequence initial state), ``mlp_decode``
(B=64, H=12, d=64, hidden 256, 256 single-token steps) and ``linear_few_heads`` (B=1, H=4, d=64,
T=16384, b=16: a batch-1 prompt with few heads, where the split along the sequence pays).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    d: int
    chunk: int
    dtype: str  # "f32" or "bf16": dtype of Q, K, V and Z
    seed: int
    hidden: int = 0  # TTT-MLP inner width (0 = TTT-Linear)
    normalize_q: bool = True
    eta_const: float | None = None
    w_zero: bool = False
    w_std: float = 0.02
    chunks: tuple = field(default_factory=tuple)  # chunk sweep, long-context workload

    @property
    def tokens(self) -> int:
        return self.B * self.T


WORKLOADS = {
    "oracle_check": Workload("oracle_check", B=1, H=1, T=64, d=16, chunk=16, dtype="f32", seed=1001,
                             normalize_q=False, eta_const=0.1, w_zero=True),
    "linear_prefill": Workload("linear_prefill", B=8, H=12, T=2048, d=64, chunk=16, dtype="bf16", seed=1002),
    "mlp_prefill": Workload("mlp_prefill", B=8, H=12, T=2048, d=64, chunk=16, dtype="bf16", seed=1003,
                            hidden=256),
    "long_context": Workload("long_context", B=1, H=16, T=32768, d=128, chunk=16, dtype="bf16", seed=1004,
                             chunks=(16, 64, 512)),
    # decode: T is the number of successive single-token steps
    "decode": Workload("decode", B=256, H=12, T=1024, d=64, chunk=1, dtype="bf16", seed=1005),
    # few heads, long sequence (batch-1 prompt): one-pass scan against the split along the sequence
    "linear_few_heads": Workload("linear_few_heads", B=1, H=4, T=16384, d=64, chunk=16, dtype="bf16", seed=1007),
    # TTT-MLP decode: 768 heads x 128 KB of fp32 state (the same 100.7 MB of state as the Linear decode)
    "mlp_decode": Workload("mlp_decode", B=64, H=12, T=256, d=64, chunk=1, dtype="bf16", seed=1006, hidden=256),
}


def torch_dtype(dtype: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def round_to(x64: np.ndarray, dtype: str) -> torch.Tensor:
    """float64 -> float32 (RN-even) -> dtype (RN-even), as a CPU torch tensor."""
    t = torch.from_numpy(np.ascontiguousarray(x64.astype(np.float32)))
    return t if dtype == "f32" else t.to(torch_dtype(dtype))


def _unit_rows(x: np.ndarray) -> np.ndarray:
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _sigmoid(u: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-u))


def draw_qkv_eta(rng, shape, d, dtype, normalize_q=True, eta_const=None):
    """Q, K, V [*shape, d] in `dtype` and eta [*shape] fp32 (CPU tensors)."""
    s = 1.0 / np.sqrt(d)
    q = rng.standard_normal(shape + (d,)) * s
    k = rng.standard_normal(shape + (d,)) * s
    v = rng.standard_normal(shape + (d,)) * s
    k = _unit_rows(k)
    if normalize_q:
        q = _unit_rows(q)
    if eta_const is not None:
        eta = np.full(shape, float(eta_const))
    else:
        eta = _sigmoid(rng.standard_normal(shape)) / d
    return round_to(q, dtype), round_to(k, dtype), round_to(v, dtype), round_to(eta, "f32")


def _weights(rng, B, H, shape, std, zero):
    if zero:
        return torch.zeros((B, H) + shape, dtype=torch.float32)
    w = round_to(rng.standard_normal((H,) + shape) * std, "f32")
    return w.unsqueeze(0).expand((B, H) + shape).contiguous()


def linear_inputs(B, H, T, d, seed, dtype="bf16", normalize_q=True, eta_const=None, w_zero=False,
                  w_std=0.02):
    """Inputs of a TTT-Linear prefill: dict of CPU tensors Q, K, V, eta, W0."""
    rng = np.random.default_rng(seed)
    Q, K, V, eta = draw_qkv_eta(rng, (B, H, T), d, dtype, normalize_q, eta_const)
    W0 = _weights(rng, B, H, (d, d), w_std, w_zero)
    return {"Q": Q, "K": K, "V": V, "eta": eta, "W0": W0}


def mlp_inputs(B, H, T, d, hidden, seed, dtype="bf16", normalize_q=True, eta_const=None, w_zero=False,
               w_std=0.02):
    """Inputs of a TTT-MLP prefill: dict of CPU tensors Q, K, V, eta, W1, W2."""
    rng = np.random.default_rng(seed)
    Q, K, V, eta = draw_qkv_eta(rng, (B, H, T), d, dtype, normalize_q, eta_const)
    W1 = _weights(rng, B, H, (d, hidden), w_std, w_zero)
    W2 = _weights(rng, B, H, (hidden, d), w_std, w_zero)
    return {"Q": Q, "K": K, "V": V, "eta": eta, "W1": W1, "W2": W2}


def decode_inputs(B, H, d, steps, seed, dtype="bf16", w_std=0.02, block=64):
    """Inputs of `steps` successive decode steps.

    Returns dict with W [B, H, d, d] fp32 (one independent draw per sequence
    and head), q, k, v [steps, B, H, d] in `dtype` and eta [steps, B, H].
    The state is drawn first, then the steps in blocks of `block` steps (each
    block draws Q, K, V, u in that order) to bound host memory.
    """
    rng = np.random.default_rng(seed)
    W = round_to(rng.standard_normal((B, H, d, d)) * w_std, "f32")
    qs, ks, vs, es = [], [], [], []
    for s0 in range(0, steps, block):
        n = min(block, steps - s0)
        q, k, v, e = draw_qkv_eta(rng, (n, B, H), d, dtype)
        qs.append(q); ks.append(k); vs.append(v); es.append(e)
    return {"W": W, "q": torch.cat(qs), "k": torch.cat(ks), "v": torch.cat(vs), "eta": torch.cat(es)}


def mlp_decode_inputs(B, H, d, hidden, steps, seed, dtype="bf16", w_std=0.02, block=64):
    """Inputs of `steps` successive TTT-MLP decode steps.

    W1 [B, H, d, hidden] then W2 [B, H, hidden, d] fp32 (one draw per sequence
    and head), then the steps in blocks of `block` (Q, K, V, u per block):
    q, k, v [steps, B, H, d] in `dtype`, eta [steps, B, H].
    """
    rng = np.random.default_rng(seed)
    W1 = round_to(rng.standard_normal((B, H, d, hidden)) * w_std, "f32")
    W2 = round_to(rng.standard_normal((B, H, hidden, d)) * w_std, "f32")
    qs, ks, vs, es = [], [], [], []
    for s0 in range(0, steps, block):
        n = min(block, steps - s0)
        q, k, v, e = draw_qkv_eta(rng, (n, B, H), d, dtype)
        qs.append(q); ks.append(k); vs.append(v); es.append(e)
    return {"W1": W1, "W2": W2, "q": torch.cat(qs), "k": torch.cat(ks), "v": torch.cat(vs), "eta": torch.cat(es)}


def backward_inputs(B, H, T, d, seed, dtype="bf16", with_dWT=True):
    """Incoming gradients of a TTT-Linear backward: dZ [B,H,T,d] ~ N(0, 1/d) in `dtype` and
    dW_T [B,H,d,d] ~ N(0, 1/d) fp32 (or None), from their own seed."""
    rng = np.random.default_rng(seed)
    s = 1.0 / np.sqrt(d)
    dZ = round_to(rng.standard_normal((B, H, T, d)) * s, dtype)
    dWT = round_to(rng.standard_normal((B, H, d, d)) * s, "f32") if with_dWT else None
    return {"dZ": dZ, "dWT": dWT}


def workload_inputs(w: Workload, chunk: int | None = None, seed_offset: int = 0):
    """Inputs of a named workload (prefill kinds)."""
    if w.hidden:
        return mlp_inputs(w.B, w.H, w.T, w.d, w.hidden, w.seed + seed_offset, w.dtype, w.normalize_q,
                          w.eta_const, w.w_zero, w.w_std)
    return linear_inputs(w.B, w.H, w.T, w.d, w.seed + seed_offset, w.dtype, w.normalize_q, w.eta_const,
                         w.w_zero, w.w_std)


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a CPU tensor (fp32 or bf16) to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
