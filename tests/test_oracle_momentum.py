"""Pins of the oracle's TTT-Linear scan with momentum (reading of the E^2-TTT article: momentum
gradient descent, squared loss, gradients at the chunk start, every token taking its own step).

What pins it, independently of the closed form written in the oracle:
  * beta = 0 is the plain scan (the oracle's pinned linear_primal);
  * chunk 1 is textbook heavy-ball SGD on 1/2 ||k W - v||^2, stepped here with torch autograd;
  * exact rational arithmetic (Python fractions) of the token-level rule on a tiny case;
  * the token-level primal and the closed-form dual agree to 1e-12;
  * (Z, W, M) are jointly linear in (W0, M0, V).
CPU only.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import oracle as O


def _inputs(B, H, T, d, seed, m0=True):
    rng = np.random.default_rng(seed)
    Q, K, V = (rng.standard_normal((B, H, T, d)) / math.sqrt(d) for _ in range(3))
    eta = rng.uniform(0.05, 0.6, (B, H, T))
    W0 = rng.standard_normal((B, H, d, d)) * 0.3
    M0 = rng.standard_normal((B, H, d, d)) * 0.2 if m0 else None
    return Q, K, V, eta, W0, M0


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


@pytest.mark.parametrize("chunk", [1, 3, 16])
def test_zero_momentum_is_the_plain_scan(chunk):
    Q, K, V, eta, W0, M0 = _inputs(2, 2, 37, 5, 60 + chunk)
    Zr, Wr = O.linear_primal(Q, K, V, eta, W0, chunk)
    for fn in (O.linear_momentum_primal, O.linear_momentum_dual):
        Z, W, _ = fn(Q, K, V, eta, W0, M0, 0.0, chunk)
        assert _rel(Z, Zr) < 1e-13 and _rel(W, Wr) < 1e-13


@pytest.mark.parametrize("beta", [0.5, 0.9])
@pytest.mark.parametrize("chunk", [1, 2, 5, 16, 64])
@pytest.mark.parametrize("m0", [True, False])
def test_primal_equals_closed_form(beta, chunk, m0):
    Q, K, V, eta, W0, M0 = _inputs(1, 3, 70, 6, 70 + chunk, m0)  # 70 tokens: ragged last chunk
    a = O.linear_momentum_primal(Q, K, V, eta, W0, M0, beta, chunk)
    b = O.linear_momentum_dual(Q, K, V, eta, W0, M0, beta, chunk)
    for x, y in zip(a, b):
        assert _rel(y, x) < 1e-12


def test_chunk_one_is_heavy_ball_sgd():
    Q, K, V, eta, W0, M0 = _inputs(1, 1, 9, 4, 80)
    beta = 0.8
    Z, W, M = O.linear_momentum_primal(Q, K, V, eta, W0, M0, beta, 1)
    Wt = torch.tensor(W0[0, 0])
    Mt = torch.tensor(M0[0, 0])
    for t in range(9):
        w = Wt.clone().requires_grad_(True)
        k, v = torch.tensor(K[0, 0, t]), torch.tensor(V[0, 0, t])
        (0.5 * ((k @ w - v) ** 2).sum()).backward()
        Mt = beta * Mt + w.grad
        Wt = Wt - eta[0, 0, t] * Mt
        assert _rel(Z[0, 0, t], (torch.tensor(Q[0, 0, t]) @ Wt).numpy()) < 1e-12
    assert _rel(W[0, 0], Wt.numpy()) < 1e-12 and _rel(M[0, 0], Mt.numpy()) < 1e-12


def test_exact_rational_case():
    # d = 2, three tokens in chunks of two, beta = 1/2, computed in exact rationals from the rule
    F = Fraction
    q = [[F(1), F(1)], [F(1), F(0)], [F(0), F(1)]]
    k = [[F(1), F(0)], [F(1), F(1)], [F(0), F(1)]]
    v = [[F(0), F(1)], [F(1), F(1)], [F(1), F(0)]]
    eta = [F(1, 2), F(1, 4), F(1, 2)]
    W = [[F(1), F(2)], [F(0), F(1)]]
    M = [[F(1, 2), F(0)], [F(0), F(-1, 2)]]
    beta = F(1, 2)
    Z = []
    for t0 in (0, 2):
        Ws = [row[:] for row in W]
        for i in range(t0, min(t0 + 2, 3)):
            e = [sum(k[i][a] * Ws[a][c] for a in range(2)) - v[i][c] for c in range(2)]
            M = [[beta * M[a][c] + k[i][a] * e[c] for c in range(2)] for a in range(2)]
            W = [[W[a][c] - eta[i] * M[a][c] for c in range(2)] for a in range(2)]
            Z.append([sum(q[i][a] * W[a][c] for a in range(2)) for c in range(2)])
    arr = lambda x: np.array(x, dtype=float)
    args = (arr(q)[None, None], arr(k)[None, None], arr(v)[None, None], arr(eta)[None, None],
            arr([[1, 2], [0, 1]])[None, None], arr([[0.5, 0], [0, -0.5]])[None, None], 0.5, 2)
    for fn in (O.linear_momentum_primal, O.linear_momentum_dual):
        z, w, m = fn(*args)
        assert np.allclose(z[0, 0], arr(Z), rtol=0, atol=1e-15)
        assert np.allclose(w[0, 0], arr(W), rtol=0, atol=1e-15)
        assert np.allclose(m[0, 0], arr(M), rtol=0, atol=1e-15)


def test_joint_linearity_in_state_momentum_and_targets():
    Q, K, V, eta, W0, M0 = _inputs(1, 2, 21, 4, 90)
    a = O.linear_momentum_dual(Q, K, V, eta, W0, M0, 0.7, 4)
    b = O.linear_momentum_dual(Q, K, -1.5 * V, eta, -1.5 * W0, -1.5 * M0, 0.7, 4)
    for x, y in zip(a, b):
        assert np.allclose(y, -1.5 * x, rtol=1e-12, atol=1e-13)
