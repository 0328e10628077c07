"""Pins of the oracle's TTT-MLP backward (the gradient of the chunked TTT-MLP scan).

The backward is written from the chain rule of the dual-form block formulas.  These tests pin it to
facts that do not go through that derivation: central finite differences of the token-level
definition (the primal scan, gradients at each block's start, read-out after the step), the second
derivative of the tanh-form GELU against finite differences of its first derivative, the
closed form of the zero-step-size case, and linearity in the incoming gradients.  CPU only.
"""
import math

import numpy as np
import pytest

from oracle import oracle as O


def _inputs(B, H, T, d, hd, seed, w_std=0.4):
    rng = np.random.default_rng(seed)
    Q, K, V = (rng.standard_normal((B, H, T, d)) / math.sqrt(d) for _ in range(3))
    eta = rng.uniform(0.05, 0.6, (B, H, T))
    W1 = rng.standard_normal((B, H, d, hd)) * w_std
    W2 = rng.standard_normal((B, H, hd, d)) * w_std
    dZ = rng.standard_normal((B, H, T, d))
    dW1T = rng.standard_normal((B, H, d, hd))
    dW2T = rng.standard_normal((B, H, hd, d))
    return Q, K, V, eta, W1, W2, dZ, dW1T, dW2T


def _fd(args, chunk, dZ, dW1T, dW2T, h=1e-5):
    """Central differences of L = sum(dZ . Z) + sum(dW1T . W1_T) + sum(dW2T . W2_T) of the primal
    scan, over every element of every input."""
    def L(*a):
        Z, W1, W2 = O.mlp_primal(*a, chunk)
        s = float(np.sum(dZ * Z))
        if dW1T is not None:
            s += float(np.sum(dW1T * W1))
        if dW2T is not None:
            s += float(np.sum(dW2T * W2))
        return s

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


@pytest.mark.parametrize("chunk", [1, 2, 3, 5])
@pytest.mark.parametrize("with_state_grad", [True, False])
def test_mlp_backward_matches_finite_differences(chunk, with_state_grad):
    # T = 5, d = 2, hidden 3: chunks 2 and 3 end with a shorter block
    Q, K, V, eta, W1, W2, dZ, dW1T, dW2T = _inputs(1, 2, 5, 2, 3, 40 + chunk)
    if not with_state_grad:
        dW1T = dW2T = None
    g = O.mlp_backward(Q, K, V, eta, W1, W2, dZ, dW1T, dW2T, chunk)
    fds = _fd([Q, K, V, eta, W1, W2], chunk, dZ, dW1T, dW2T)
    for name, ga, fa in zip(("dQ", "dK", "dV", "deta", "dW1", "dW2"), g, fds):
        assert np.max(np.abs(ga - fa)) <= 2e-7 * max(1.0, np.max(np.abs(fa))), name


def test_gelu_second_derivative_matches_finite_differences():
    for x in (-3.1, -1.0, -0.2, 0.0, 0.35, 1.7, 4.0):
        h = 1e-5
        fd = (O.gelu_prime(x + h) - O.gelu_prime(x - h)) / (2 * h)
        assert abs(O.gelu_second(x) - fd) <= 1e-8, x


def test_mlp_backward_with_zero_step_size():
    # eta = 0: Z = GELU(Q W1) W2 and the state does not move, so with P = dZ W2^T . GELU'(Q W1):
    # dQ = P W1^T, dK = dV = 0, dW1 = Q^T P + dW1T, dW2 = GELU(Q W1)^T dZ + dW2T
    Q, K, V, eta, W1, W2, dZ, dW1T, dW2T = _inputs(2, 1, 9, 3, 5, 50)
    eta = np.zeros_like(eta)
    dQ, dK, dV, deta, dW1, dW2 = O.mlp_backward(Q, K, V, eta, W1, W2, dZ, dW1T, dW2T, 4)
    U = Q @ W1
    g = np.vectorize(O.gelu)(U)
    gp = np.vectorize(O.gelu_prime)(U)
    P = (dZ @ np.swapaxes(W2, -1, -2)) * gp
    assert np.allclose(dQ, P @ np.swapaxes(W1, -1, -2), atol=1e-12)
    assert np.all(dK == 0) and np.all(dV == 0)
    assert np.allclose(dW1, np.swapaxes(Q, -1, -2) @ P + dW1T, atol=1e-12)
    assert np.allclose(dW2, np.swapaxes(g, -1, -2) @ dZ + dW2T, atol=1e-12)


def test_mlp_backward_is_linear_in_the_incoming_gradients():
    Q, K, V, eta, W1, W2, dZ, dW1T, dW2T = _inputs(1, 2, 8, 3, 4, 51)
    g1 = O.mlp_backward(Q, K, V, eta, W1, W2, dZ, dW1T, dW2T, 3)
    g2 = O.mlp_backward(Q, K, V, eta, W1, W2, 1.5 * dZ, 1.5 * dW1T, 1.5 * dW2T, 3)
    for a, b in zip(g1, g2):
        assert np.allclose(b, 1.5 * a, rtol=1e-12, atol=1e-13)
