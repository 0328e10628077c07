"""Shared helpers of the GPU parity tests: tolerances, error metric, device moves."""
import numpy as np
import torch

from test_sequence_layers_07_b300 import workloads as WL

# Tolerances on max|delta| / ||ref||_inf, per output (Z and each final weight matrix):
# 1e-4 for fp32 inputs and 2e-2 for bf16 inputs.
TOL = {"f32": 1e-4, "bf16": 2e-2}


def rel_err(got: torch.Tensor, ref: np.ndarray) -> float:
    g = got.detach().to("cpu", torch.float64).numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), "non-finite values in the GPU result"
    den = float(np.max(np.abs(ref)))
    return float(np.max(np.abs(g - ref)) / (den if den > 0 else 1.0))


def cuda(d: dict) -> dict:
    return {k: v.cuda() for k, v in d.items()}


def f64(d: dict) -> dict:
    return {k: WL.to_f64(v) for k, v in d.items()}


def heads(x: dict, idx):
    """Select (batch, head) pairs idx = [(b, h), ...] from a dict of [B,H,...] arrays -> [1, n, ...]."""
    return {k: np.stack([v[b, h] for (b, h) in idx])[None] for k, v in x.items()}
