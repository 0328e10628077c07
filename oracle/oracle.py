"""Python binding of the fp64 CPU oracle (``ttt_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library never
imports this module and has no fallback to it.

Every function takes float64 numpy arrays in the row-major layouts of the C
file and returns new float64 arrays; inputs are not modified (except that
``linear_decode`` returns the updated state rather than writing into W).

What each routine computes, and the page passages it follows, is stated in the
header of ``ttt_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ttt_oracle.c")
_LIB = os.path.join(_HERE, "_ttt_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``ttt_oracle.c`` into ``_ttt_oracle.so`` with gcc (fp64, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", _LIB, "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            i = ctypes.c_int
            sig5 = [dp] * 7 + [i] * 5
            for name in ("oracle_linear_primal", "oracle_linear_dual"):
                f = getattr(lib, name)
                f.argtypes = sig5
                f.restype = None
            for name in ("oracle_mlp_primal", "oracle_mlp_dual"):
                f = getattr(lib, name)
                f.argtypes = [dp] * 9 + [i] * 6
                f.restype = None
            lib.oracle_linear_backward.argtypes = [dp] * 12 + [i] * 5
            lib.oracle_linear_backward.restype = None
            lib.oracle_mlp_backward.argtypes = [dp] * 15 + [i] * 6
            lib.oracle_mlp_backward.restype = None
            lib.oracle_gelu_second.argtypes = [ctypes.c_double]
            lib.oracle_gelu_second.restype = ctypes.c_double
            for name in ("oracle_linear_momentum_primal", "oracle_linear_momentum_dual"):
                f = getattr(lib, name)
                f.argtypes = [dp] * 6 + [ctypes.c_double] + [dp] * 3 + [i] * 5
                f.restype = None
            lib.oracle_linear_decode.argtypes = [dp] * 6 + [i] * 3
            lib.oracle_linear_decode.restype = None
            lib.oracle_mlp_token_grad.argtypes = [dp] * 7 + [i] * 2
            lib.oracle_mlp_token_grad.restype = ctypes.c_double
            lib.oracle_mlp_forward.argtypes = [dp] * 4 + [i] * 2
            lib.oracle_mlp_forward.restype = None
            lib.oracle_gelu.argtypes = [ctypes.c_double]
            lib.oracle_gelu.restype = ctypes.c_double
            lib.oracle_gelu_prime.argtypes = [ctypes.c_double]
            lib.oracle_gelu_prime.restype = ctypes.c_double
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = i
            lib.oracle_set_num_threads.argtypes = [i]
            lib.oracle_set_num_threads.restype = None
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def gelu(x: float) -> float:
    return _load().oracle_gelu(float(x))


def gelu_prime(x: float) -> float:
    return _load().oracle_gelu_prime(float(x))


def _linear(fn_name, Q, K, V, eta, W0, chunk):
    Q, K, V, eta, W0 = (_f64(a) for a in (Q, K, V, eta, W0))
    B, H, T, d = Q.shape
    assert K.shape == V.shape == Q.shape and eta.shape == (B, H, T) and W0.shape == (B, H, d, d)
    assert 1 <= chunk
    Z = np.zeros_like(Q)
    W = np.zeros_like(W0)
    getattr(_load(), fn_name)(_p(Q), _p(K), _p(V), _p(eta), _p(W0), _p(Z), _p(W), B, H, T, d, int(chunk))
    return Z, W


def linear_primal(Q, K, V, eta, W0, chunk):
    """Token-level TTT-Linear scan (gradients at each block's start). Returns (Z, W_final)."""
    return _linear("oracle_linear_primal", Q, K, V, eta, W0, chunk)


def linear_dual(Q, K, V, eta, W0, chunk):
    """Dual (matrix) form of the same scan. Returns (Z, W_final)."""
    return _linear("oracle_linear_dual", Q, K, V, eta, W0, chunk)


def _momentum(fn_name, Q, K, V, eta, W0, M0, beta, chunk):
    Q, K, V, eta, W0 = (_f64(a) for a in (Q, K, V, eta, W0))
    B, H, T, d = Q.shape
    assert K.shape == V.shape == Q.shape and eta.shape == (B, H, T) and W0.shape == (B, H, d, d) and chunk >= 1
    Mp = None
    if M0 is not None:
        M0 = _f64(M0)
        assert M0.shape == W0.shape
        Mp = _p(M0)
    Z, W, M = np.zeros_like(Q), np.zeros_like(W0), np.zeros_like(W0)
    getattr(_load(), fn_name)(_p(Q), _p(K), _p(V), _p(eta), _p(W0), Mp, float(beta), _p(Z), _p(W), _p(M),
                              B, H, T, d, int(chunk))
    return Z, W, M


def linear_momentum_primal(Q, K, V, eta, W0, M0, beta, chunk):
    """Token-level TTT-Linear scan with momentum (gradients at each chunk's start; M0 None = zero).
    Returns (Z, W_final, M_final)."""
    return _momentum("oracle_linear_momentum_primal", Q, K, V, eta, W0, M0, beta, chunk)


def linear_momentum_dual(Q, K, V, eta, W0, M0, beta, chunk):
    """Closed (dual) form of the same scan. Returns (Z, W_final, M_final)."""
    return _momentum("oracle_linear_momentum_dual", Q, K, V, eta, W0, M0, beta, chunk)


def linear_backward(Q, K, V, eta, W0, dZ, dWT, chunk):
    """Gradient of the TTT-Linear scan with respect to (Q, K, V, eta, W0), given the gradients dZ
    of the outputs and dWT of the final state (None: zero).  Returns (dQ, dK, dV, deta, dW0)."""
    Q, K, V, eta, W0, dZ = (_f64(a) for a in (Q, K, V, eta, W0, dZ))
    B, H, T, d = Q.shape
    assert K.shape == V.shape == dZ.shape == Q.shape and eta.shape == (B, H, T) and W0.shape == (B, H, d, d)
    assert 1 <= chunk
    dWT_p = None
    if dWT is not None:
        dWT = _f64(dWT)
        assert dWT.shape == W0.shape
        dWT_p = _p(dWT)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(Q), np.zeros_like(Q)
    deta = np.zeros_like(eta)
    dW0 = np.zeros_like(W0)
    _load().oracle_linear_backward(_p(Q), _p(K), _p(V), _p(eta), _p(W0), _p(dZ), dWT_p, _p(dQ), _p(dK), _p(dV),
                                   _p(deta), _p(dW0), B, H, T, d, int(chunk))
    return dQ, dK, dV, deta, dW0


def _mlp(fn_name, Q, K, V, eta, W1, W2, chunk):
    Q, K, V, eta, W1, W2 = (_f64(a) for a in (Q, K, V, eta, W1, W2))
    B, H, T, d = Q.shape
    hd = W1.shape[-1]
    assert W1.shape == (B, H, d, hd) and W2.shape == (B, H, hd, d) and eta.shape == (B, H, T)
    Z = np.zeros_like(Q)
    W1o = np.zeros_like(W1)
    W2o = np.zeros_like(W2)
    getattr(_load(), fn_name)(_p(Q), _p(K), _p(V), _p(eta), _p(W1), _p(W2), _p(Z), _p(W1o), _p(W2o),
                              B, H, T, d, hd, int(chunk))
    return Z, W1o, W2o


def mlp_primal(Q, K, V, eta, W1, W2, chunk):
    """Token-level TTT-MLP scan. Returns (Z, W1_final, W2_final)."""
    return _mlp("oracle_mlp_primal", Q, K, V, eta, W1, W2, chunk)


def mlp_dual(Q, K, V, eta, W1, W2, chunk):
    """Dual form of the TTT-MLP scan. Returns (Z, W1_final, W2_final)."""
    return _mlp("oracle_mlp_dual", Q, K, V, eta, W1, W2, chunk)


def mlp_backward(Q, K, V, eta, W1, W2, dZ, dW1T, dW2T, chunk):
    """Gradient of the TTT-MLP scan with respect to (Q, K, V, eta, W1_0, W2_0), given dZ and the
    gradients dW1T, dW2T of the final state (None: zero).  Returns (dQ, dK, dV, deta, dW1, dW2)."""
    Q, K, V, eta, W1, W2, dZ = (_f64(a) for a in (Q, K, V, eta, W1, W2, dZ))
    B, H, T, d = Q.shape
    hd = W1.shape[-1]
    assert K.shape == V.shape == dZ.shape == Q.shape and eta.shape == (B, H, T)
    assert W1.shape == (B, H, d, hd) and W2.shape == (B, H, hd, d) and chunk >= 1
    ptrs = []
    for g, ref in ((dW1T, W1), (dW2T, W2)):
        if g is None:
            ptrs.append(None)
        else:
            g = _f64(g)
            assert g.shape == ref.shape
            ptrs.append(g)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(Q), np.zeros_like(Q)
    deta = np.zeros_like(eta)
    dW1, dW2 = np.zeros_like(W1), np.zeros_like(W2)
    _load().oracle_mlp_backward(_p(Q), _p(K), _p(V), _p(eta), _p(W1), _p(W2), _p(dZ),
                                None if ptrs[0] is None else _p(ptrs[0]), None if ptrs[1] is None else _p(ptrs[1]),
                                _p(dQ), _p(dK), _p(dV), _p(deta), _p(dW1), _p(dW2), B, H, T, d, hd, int(chunk))
    return dQ, dK, dV, deta, dW1, dW2


def gelu_second(x: float) -> float:
    return _load().oracle_gelu_second(float(x))


def linear_decode(q, k, v, eta, W):
    """One online TTT-Linear step for every (batch, head). Returns (z, W_new)."""
    q, k, v, eta = (_f64(a) for a in (q, k, v, eta))
    Wn = _f64(W).copy()
    B, H, d = q.shape
    assert eta.shape == (B, H) and Wn.shape == (B, H, d, d)
    z = np.zeros_like(q)
    _load().oracle_linear_decode(_p(q), _p(k), _p(v), _p(eta), _p(Wn), _p(z), B, H, d)
    return z, Wn


def mlp_decode(q, k, v, eta, W1, W2):
    """One online TTT-MLP step for every (batch, head): the token-level scan on a
    single token (block of one).  q,k,v [B,H,d], eta [B,H]; returns (z, W1_new, W2_new)."""
    q, k, v, eta = (_f64(a) for a in (q, k, v, eta))
    Z, A, Bm = mlp_primal(q[:, :, None], k[:, :, None], v[:, :, None], eta[:, :, None], W1, W2, 1)
    return Z[:, :, 0], A, Bm


def mlp_token_grad(k, v, W1, W2):
    """Loss and chain-rule pieces (a, e1, e2) of 1/2||GELU(kW1)W2 - v||^2 for one token.

    The gradients are dW1 = outer(k, e1) and dW2 = outer(a, e2).
    """
    k, v, W1, W2 = (_f64(a) for a in (k, v, W1, W2))
    d, hd = W1.shape
    a = np.zeros(hd)
    e1 = np.zeros(hd)
    e2 = np.zeros(d)
    loss = _load().oracle_mlp_token_grad(_p(k), _p(v), _p(W1), _p(W2), _p(a), _p(e1), _p(e2), d, hd)
    return loss, a, e1, e2


def mlp_forward(x, W1, W2):
    """f(x; W1, W2) = GELU(x W1) W2 for one row x."""
    x, W1, W2 = (_f64(a) for a in (x, W1, W2))
    d, hd = W1.shape
    y = np.zeros(d)
    _load().oracle_mlp_forward(_p(x), _p(W1), _p(W2), _p(y), d, hd)
    return y
