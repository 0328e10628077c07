"""Shared helpers of the GPU parity tests: tolerances, error metric, device moves, and the record
of observed error margins."""
import json
import os
import threading

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


class Margins:
    """Observed max|delta| / ||ref||_inf of the full-size workload checks, written as JSON to the
    path in TTT_PARITY_MARGINS (if set) when the test session ends."""

    def __init__(self):
        self._lock = threading.Lock()
        self.rows = {}

    def record(self, name: str, tol: float, **errs: float) -> None:
        with self._lock:
            self.rows[name] = {"tol": tol, **{k: float(v) for k, v in errs.items()}}

    def dump(self) -> None:
        path = os.environ.get("TTT_PARITY_MARGINS")
        if not path or not self.rows:
            return
        old = {}
        if os.path.exists(path):
            try:
                old = json.load(open(path))
            except ValueError:
                old = {}
        old.update(self.rows)
        os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
        with open(path, "w") as f:
            json.dump(old, f, indent=1, sort_keys=True)


MARGINS = Margins()


def check(name: str, tol: float, **pairs):
    """Compare each (got, ref) pair, record the errors under `name`, and assert every one <= tol."""
    errs = {k: rel_err(g, r) for k, (g, r) in pairs.items()}
    MARGINS.record(name, tol, **errs)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{name}: {bad} above {tol}"
    return errs
