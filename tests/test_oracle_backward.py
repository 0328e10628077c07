"""Pins of the oracle's TTT-Linear backward (the gradient of the chunked scan).

The backward is written from the chain rule of the dual-form block formulas.  These tests pin it
to facts that do not go through that derivation: central finite differences of the token-level
definition (the primal scan), closed forms of two special cases, and linearity in the incoming
gradients.  CPU only.
"""
import math

import numpy as np
import pytest

from oracle import oracle as O


def _inputs(B, H, T, d, seed):
    rng = np.random.default_rng(seed)
    Q, K, V = (rng.standard_normal((B, H, T, d)) / math.sqrt(d) for _ in range(3))
    eta = rng.uniform(0.05, 0.6, (B, H, T))
    W0 = rng.standard_normal((B, H, d, d)) * 0.3
    dZ = rng.standard_normal((B, H, T, d))
    dWT = rng.standard_normal((B, H, d, d))
    return Q, K, V, eta, W0, dZ, dWT


def _fd(args, chunk, dZ, dWT, h=1e-5):
    """Central differences of L = sum(dZ . Z) + sum(dWT . W_T) over every input element."""
    def L(*a):
        Z, W = O.linear_primal(*a, chunk)
        return float(np.sum(dZ * Z) + (np.sum(dWT * W) if dWT is not None else 0.0))

    out = []
    for ai, a in enumerate(args):
        fd = np.zeros_like(a)
        for idx in np.ndindex(a.shape):
            ap = [x.copy() for x in args]
            am = [x.copy() for x in args]
            ap[ai][idx] += h
            am[ai][idx] -= h
            fd[idx] = (L(*ap) - L(*am)) / (2 * h)
        out.append(fd)
    return out


@pytest.mark.parametrize("chunk", [1, 2, 3, 4, 7])
@pytest.mark.parametrize("with_dWT", [True, False])
def test_backward_matches_finite_differences(chunk, with_dWT):
    # T = 7: chunks 2, 3 and 4 end with a shorter block
    Q, K, V, eta, W0, dZ, dWT = _inputs(1, 2, 7, 3, 20 + chunk)
    dWT = dWT if with_dWT else None
    g = O.linear_backward(Q, K, V, eta, W0, dZ, dWT, chunk)
    for name, ga, fa in zip(("dQ", "dK", "dV", "deta", "dW0"), g, _fd([Q, K, V, eta, W0], chunk, dZ, dWT)):
        assert np.max(np.abs(ga - fa)) <= 1e-7 * max(1.0, np.max(np.abs(fa))), name


def test_backward_with_zero_step_size():
    # eta = 0: Z = Q W0 and W_T = W0, so dQ = dZ W0^T, dK = dV = 0, dW0 = sum_t q_t^T dz_t + dWT
    Q, K, V, eta, W0, dZ, dWT = _inputs(2, 2, 12, 4, 31)
    eta = np.zeros_like(eta)
    dQ, dK, dV, deta, dW0 = O.linear_backward(Q, K, V, eta, W0, dZ, dWT, 4)
    assert np.allclose(dQ, dZ @ np.swapaxes(W0, -1, -2), atol=1e-13)
    assert np.all(dK == 0) and np.all(dV == 0)
    assert np.allclose(dW0, np.swapaxes(Q, -1, -2) @ dZ + dWT, atol=1e-12)


def test_backward_single_block_state_only():
    # one block, dZ = 0: W_T = (I - K^T D K) W0 + K^T D V, so dW0 = (I - K^T D K) dWT (symmetric
    # factor) and dV = D K dWT
    Q, K, V, eta, W0, dZ, dWT = _inputs(1, 1, 6, 3, 32)
    dZ = np.zeros_like(dZ)
    dQ, dK, dV, deta, dW0 = O.linear_backward(Q, K, V, eta, W0, dZ, dWT, 6)
    k, D = K[0, 0], np.diag(eta[0, 0])
    assert np.allclose(dW0[0, 0], (np.eye(3) - k.T @ D @ k) @ dWT[0, 0], atol=1e-13)
    assert np.allclose(dV[0, 0], D @ k @ dWT[0, 0], atol=1e-13)
    assert np.all(dQ == 0)


def test_backward_is_linear_in_the_incoming_gradients():
    Q, K, V, eta, W0, dZ, dWT = _inputs(1, 2, 10, 3, 33)
    g1 = O.linear_backward(Q, K, V, eta, W0, dZ, dWT, 4)
    g2 = O.linear_backward(Q, K, V, eta, W0, -2.5 * dZ, -2.5 * dWT, 4)
    for a, b in zip(g1, g2):
        assert np.allclose(b, -2.5 * a, rtol=1e-12, atol=1e-13)
