"""The oracle's pins catch plausible mistakes.

Each mutant below plants one plausible bug in a copy of ``oracle/ttt_oracle.c``
(a dropped term, a wrong sign, a wrong token index, a transposed operand, the
gradient taken at the wrong state, a wrong constant).  The copy is compiled
with gcc into a temporary library and bound through a fresh instance of
``oracle/oracle.py``.  The test asserts that at least one pin fails on every
mutant, and that every pin passes on the unmodified source: a pin set that a
mutant survives would not be evidence that the oracle is right.

The pins used here are the same facts as ``test_oracle_pins.py`` (hand-derived
d = 2 examples, closed forms, invariants, finite differences, GELU against
torch), restated against a module argument.  Everything runs on the CPU.
"""
import importlib.util
import json
import math
import os

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ttt_oracle.c")
BINDING = os.path.join(ROOT, "oracle", "oracle.py")
GOLDEN = os.path.join(ROOT, "tests", "golden", "linear_d2_hand.json")

# (name, text in ttt_oracle.c, replacement); each text must occur exactly once
MUTANTS = [
    ("dual mask drops the diagonal", "A[(size_t)i * n + j] = (j <= i) ?", "A[(size_t)i * n + j] = (j < i) ?"),
    ("dual scores use the query token's eta", "? ec[j] * dot(Qc + (size_t)i * d, Kc", "? ec[i] * dot(Qc + (size_t)i * d, Kc"),
    ("dual error sign flipped", "E[(size_t)i * d + c] -= Vc[(size_t)i * d + c];",
     "E[(size_t)i * d + c] += Vc[(size_t)i * d + c];"),
    ("dual update transposed", "rank1_sub(Wn, ec[j], Kc + (size_t)j * d, E + (size_t)j * d, d, d);",
     "rank1_sub(Wn, ec[j], E + (size_t)j * d, Kc + (size_t)j * d, d, d);"),
    ("dual update with reversed step sizes", "rank1_sub(Wn, ec[j], Kc + (size_t)j * d, E + (size_t)j * d, d, d);",
     "rank1_sub(Wn, ec[n - 1 - j], Kc + (size_t)j * d, E + (size_t)j * d, d, d);"),
    ("primal gradient at the running state", "oracle_linear_token_error(k, V + (size_t)i * d, Ws, e, d); /* at Ws */",
     "oracle_linear_token_error(k, V + (size_t)i * d, W, e, d); /* at Ws */"),
    ("primal readout before the step", "vecmat(Q + (size_t)i * d, W, Z + (size_t)i * d, d, d);     /* readout */",
     "vecmat(Q + (size_t)i * d, Ws, Z + (size_t)i * d, d, d);     /* readout */"),
    ("loss without the factor 1/2", "    for (int j = 0; j < d; ++j) e[j] -= v[j];\n}",
     "    for (int j = 0; j < d; ++j) e[j] = 2.0 * (e[j] - v[j]);\n}"),
    ("GELU cubic coefficient", "GELU_A = 0.044715;", "GELU_A = 0.04715;"),
    ("GELU' drops the chain-rule term", "return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * dinner;",
     "return 0.5 * (1.0 + t);"),
    ("MLP activation dropped", "for (int m = 0; m < hd; ++m) a[m] = oracle_gelu(u[m]);",
     "for (int m = 0; m < hd; ++m) a[m] = u[m];"),
    ("MLP backprop drops GELU'", "e1[m] = s * oracle_gelu_prime(u[m]);", "e1[m] = s;"),
    ("MLP dual layer-1 delta dropped", "for (int m = 0; m < hd; ++m) hq[m] -= a1 * e1[m];",
     "for (int m = 0; m < hd; ++m) hq[m] -= 0.0 * a1 * e1[m];"),
    ("MLP dual layer-2 scores use Hk for Hq", "double a2 = ec[j] * dot(hq, Hk + (size_t)j * hd, hd);",
     "double a2 = ec[j] * dot(Hk + (size_t)i * hd, Hk + (size_t)j * hd, hd);"),
    ("MLP dual W1 update reads Q", "rank1_sub(W1n, ec[j], Kc + (size_t)j * d, E1 + (size_t)j * hd, d, hd);",
     "rank1_sub(W1n, ec[j], Qc + (size_t)j * d, E1 + (size_t)j * hd, d, hd);"),
    ("MLP dual error sign flipped", "for (int c = 0; c < d; ++c) e2[c] -= Vc[(size_t)i * d + c];",
     "for (int c = 0; c < d; ++c) e2[c] += Vc[(size_t)i * d + c];"),
    ("MLP primal W2 step uses the pre-activation", "rank1_sub(W2, eta[i], a, e2, hd, d);  /* W2 -= eta a^T e2 */",
     "rank1_sub(W2, eta[i], e1, e2, hd, d);  /* W2 -= eta a^T e2 */"),
    ("backward dE drops the read-out term", "for (int i = j; i < b; ++i) acc -= S[(size_t)i * b + j] * ec[j]",
     "for (int i = j; i < b; ++i) acc -= 0.0 * S[(size_t)i * b + j] * ec[j]"),
    ("backward dK drops the state-update term", "acc -= ec[j] * dot(E + (size_t)j * d, dW + (size_t)k * d, d);",
     "acc -= 0.0 * ec[j] * dot(E + (size_t)j * d, dW + (size_t)k * d, d);"),
    ("backward deta update term sign", "double de = -dot(E + (size_t)j * d, KdW + (size_t)j * d, d);",
     "double de = dot(E + (size_t)j * d, KdW + (size_t)j * d, d);"),
    ("backward mask drops the diagonal", "dA[(size_t)i * b + j] = (j <= i) ?", "dA[(size_t)i * b + j] = (j < i) ?"),
    ("backward dW drops K^T dE", "rank1_sub(dWp, -1.0, Kc + (size_t)i * d, dE + (size_t)i * d, d, d);",
     "rank1_sub(dWp, -0.0, Kc + (size_t)i * d, dE + (size_t)i * d, d, d);"),
    ("backward uses the state after the block",
     "const double *W = Ws + (size_t)n * dd; /* the state at the start of block n */",
     "const double *W = Ws + (size_t)(n + 1) * dd; /* the state at the start of block n */"),
    ("backward dQ scores term uses the query's eta", "acc += dA[(size_t)i * b + j] * ec[j] * Kc[(size_t)j * d + k];",
     "acc += dA[(size_t)i * b + j] * ec[i] * Kc[(size_t)j * d + k];"),
    ("MLP backward drops GELU''", "dZk[at] = dE1[at] * Gk[at] * oracle_gelu_second(Zk[at]);",
     "dZk[at] = 0.0 * dE1[at] * Gk[at] * oracle_gelu_second(Zk[at]);"),
    ("GELU'' sign of the tanh term", "return s * u1 + 0.5 * x * s * (u2 - 2.0 * t * u1 * u1);",
     "return s * u1 + 0.5 * x * s * (u2 + 2.0 * t * u1 * u1);"),
    ("MLP backward layer-2 scores mask drops the diagonal",
     "dA2[(size_t)i * b + j] = (j <= i) ? -dot(dZc + (size_t)i * d, E2 + (size_t)j * d, d) : 0.0;",
     "dA2[(size_t)i * b + j] = (j < i) ? -dot(dZc + (size_t)i * d, E2 + (size_t)j * d, d) : 0.0;"),
    ("MLP backward dW2 from the read-out uses Hk",
     "for (int i = 0; i < b; ++i) rank1_sub(dW2, -1.0, Hq + (size_t)i * hd, dZc + (size_t)i * d, hd, d);",
     "for (int i = 0; i < b; ++i) rank1_sub(dW2, -1.0, Hk + (size_t)i * hd, dZc + (size_t)i * d, hd, d);"),
    ("MLP backward drops dGk^T E2 in dW2",
     "for (int j = 0; j < b; ++j) rank1_sub(dW2, -1.0, dGk + (size_t)j * hd, E2 + (size_t)j * d, hd, d);",
     "for (int j = 0; j < b; ++j) rank1_sub(dW2, -0.0, dGk + (size_t)j * hd, E2 + (size_t)j * d, hd, d);"),
    ("momentum closed form: c without the token's own beta power", "bp *= beta;\n            acc += ec[i] * bp;",
     "acc += ec[i] * bp;\n            bp *= beta;"),
    ("momentum closed form scales by the key's eta", "g += ec[i] * bl;  /* adds eta_i beta^(i-j) */",
     "g += ec[j] * bl;  /* adds eta_i beta^(i-j) */"),
    ("momentum closed form: chunk-end momentum not decayed", "for (size_t x = 0; x < dd; ++x) Mn[x] = bn * M[x];",
     "for (size_t x = 0; x < dd; ++x) Mn[x] = M[x];"),
    ("momentum primal without the decay", "for (size_t x = 0; x < dd; ++x) M[x] *= beta;",
     "for (size_t x = 0; x < dd; ++x) M[x] *= 1.0;"),
    ("MLP backward layer-1 scores use the query's eta", "double a1 = ec[j] * S1[(size_t)i * b + j];\n                for (int m = 0; m < hd; ++m) dE1",
     "double a1 = ec[i] * S1[(size_t)i * b + j];\n                for (int m = 0; m < hd; ++m) dE1"),
]


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _lin(B, H, T, d, seed):
    rng = np.random.default_rng(seed)
    Q, K, V = (rng.standard_normal((B, H, T, d)) / math.sqrt(d) for _ in range(3))
    return Q, K, V, rng.uniform(0.05, 0.6, (B, H, T)), rng.standard_normal((B, H, d, d)) * 0.3


def _mlp(B, H, T, d, hd, seed):
    rng = np.random.default_rng(seed)
    Q, K, V = (rng.standard_normal((B, H, T, d)) / math.sqrt(d) for _ in range(3))
    eta = rng.uniform(0.05, 0.5, (B, H, T))
    return Q, K, V, eta, rng.standard_normal((B, H, d, hd)) * 0.5, rng.standard_normal((B, H, hd, d)) * 0.5


def _gelu_t(x):
    return torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()


# ------------------------------------------------------------ pins on a module

def pin_golden(M):
    g = json.load(open(GOLDEN))
    inp = g["inputs"]
    q, k, v = (np.array(inp[n], float)[None, None] for n in ("q", "k", "v"))
    for case in g["cases"]:
        W0 = np.array(inp["W0"], float) if case["W0"] == "inputs" else np.zeros((2, 2))
        eta = np.array(case["eta"], float)[None, None]
        for f in (M.linear_primal, M.linear_dual):
            Z, W = f(q, k, v, eta, W0[None, None], case["chunk"])
            if not (np.allclose(Z[0, 0], case["Z"], rtol=0, atol=1e-15) and
                    np.allclose(W[0, 0], case["W"], rtol=0, atol=1e-15)):
                return False
    return True


def pin_primal_dual(M):
    Q, K, V, eta, W0 = _lin(1, 2, 21, 5, 1)
    Zp, Wp = M.linear_primal(Q, K, V, eta, W0, 5)
    Zd, Wd = M.linear_dual(Q, K, V, eta, W0, 5)
    Q, K, V, eta, W1, W2 = _mlp(1, 1, 11, 4, 7, 2)
    a = M.mlp_primal(Q, K, V, eta, W1, W2, 3)
    b = M.mlp_dual(Q, K, V, eta, W1, W2, 3)
    return _rel(Zd, Zp) < 1e-12 and _rel(Wd, Wp) < 1e-12 and all(_rel(y, x) < 1e-12 for x, y in zip(a, b))


def pin_linear_attention(M):
    Q, K, V, eta, _ = _lin(1, 1, 12, 4, 3)
    S = Q[0, 0] @ K[0, 0].T
    Zla = np.array([sum(eta[0, 0, j] * S[i, j] * V[0, 0, j] for j in range(i + 1)) for i in range(12)])
    for f in (M.linear_primal, M.linear_dual):
        Z, _ = f(Q, K, V, eta, np.zeros((1, 1, 4, 4)), 12)
        if _rel(Z[0, 0], Zla) > 1e-12:
            return False
    return True


def pin_delta_rule(M):
    Q, K, V, eta, W0 = _lin(1, 1, 9, 4, 4)
    for f in (M.linear_primal, M.linear_dual):
        Z, W = f(Q, K, V, eta, W0, 1)
        Wt = W0[0, 0].copy()
        for t in range(9):
            k, v = K[0, 0, t], V[0, 0, t]
            Wt = (np.eye(4) - eta[0, 0, t] * np.outer(k, k)) @ Wt + eta[0, 0, t] * np.outer(k, v)
            if _rel(Z[0, 0, t], Q[0, 0, t] @ Wt) > 1e-12:
                return False
        if _rel(W[0, 0], Wt) > 1e-12:
            return False
    return True


def pin_consistent_targets(M):
    Q, K, _, eta, W0 = _lin(1, 1, 16, 4, 5)
    for f in (M.linear_primal, M.linear_dual):
        Z, W = f(Q, K, K @ W0, eta, W0, 4)
        if _rel(W, W0) > 1e-13 or _rel(Z, Q @ W0) > 1e-13:
            return False
    Q, K, V, eta, W1, W2 = _mlp(1, 1, 8, 4, 6, 6)
    V2 = _gelu_t(K @ W1) @ W2
    for f in (M.mlp_primal, M.mlp_dual):
        Z, A, Bm = f(Q, K, V2, eta, W1, W2, 4)
        if _rel(A, W1) > 1e-12 or _rel(Bm, W2) > 1e-12 or _rel(Z, _gelu_t(Q @ W1) @ W2) > 1e-12:
            return False
    return True


def pin_mlp_kernelised_attention(M):
    Q, K, V, eta, W1, _ = _mlp(1, 1, 7, 4, 6, 7)
    Hq, Hk = _gelu_t(Q[0, 0] @ W1[0, 0]), _gelu_t(K[0, 0] @ W1[0, 0])
    Zexp = np.array([sum(eta[0, 0, j] * (Hq[i] @ Hk[j]) * V[0, 0, j] for j in range(i + 1)) for i in range(7)])
    for f in (M.mlp_primal, M.mlp_dual):
        Z, A, Bm = f(Q, K, V, eta, W1, np.zeros((1, 1, 6, 4)), 7)
        if _rel(Z[0, 0], Zexp) > 1e-12 or _rel(A, W1) > 1e-14:
            return False
        if _rel(Bm[0, 0], Hk.T @ np.diag(eta[0, 0]) @ V[0, 0]) > 1e-12:
            return False
    return True


def pin_mlp_finite_differences(M):
    rng = np.random.default_rng(8)
    d, hd = 3, 5
    k, v = rng.standard_normal(d), rng.standard_normal(d)
    W1, W2 = rng.standard_normal((d, hd)) * 0.5, rng.standard_normal((hd, d)) * 0.5
    _, a, e1, e2 = M.mlp_token_grad(k, v, W1, W2)
    loss = lambda A, Bm: M.mlp_token_grad(k, v, A, Bm)[0]
    h = 1e-6
    fd1 = np.zeros_like(W1)
    for i in range(d):
        for m in range(hd):
            P, Mi = W1.copy(), W1.copy()
            P[i, m] += h
            Mi[i, m] -= h
            fd1[i, m] = (loss(P, W2) - loss(Mi, W2)) / (2 * h)
    fd2 = np.zeros_like(W2)
    for m in range(hd):
        for c in range(d):
            P, Mi = W2.copy(), W2.copy()
            P[m, c] += h
            Mi[m, c] -= h
            fd2[m, c] = (loss(W1, P) - loss(W1, Mi)) / (2 * h)
    y = _gelu_t(k[None] @ W1)[0] @ W2
    return (_rel(np.outer(k, e1), fd1) < 1e-6 and _rel(np.outer(a, e2), fd2) < 1e-6 and
            abs(loss(W1, W2) - 0.5 * np.sum((y - v) ** 2)) < 1e-12)


def pin_gelu(M):
    xs = torch.linspace(-5, 5, 41, dtype=torch.float64, requires_grad=True)
    y = torch.nn.functional.gelu(xs, approximate="tanh")
    y.sum().backward()
    g = np.array([M.gelu(float(x)) for x in xs.detach()])
    gp = np.array([M.gelu_prime(float(x)) for x in xs.detach()])
    return np.max(np.abs(g - y.detach().numpy())) < 1e-13 and np.max(np.abs(gp - xs.grad.numpy())) < 1e-13


def pin_mlp_online_gd(M):
    Q, K, V, eta, W1, W2 = _mlp(1, 1, 4, 3, 5, 9)
    Z, A1, A2 = M.mlp_primal(Q, K, V, eta, W1, W2, 1)
    A, Bm = W1[0, 0].copy(), W2[0, 0].copy()
    for t in range(4):
        k, v = torch.tensor(K[0, 0, t]), torch.tensor(V[0, 0, t])
        At, Bt = torch.tensor(A, requires_grad=True), torch.tensor(Bm, requires_grad=True)
        loss = 0.5 * ((torch.nn.functional.gelu(k @ At, approximate="tanh") @ Bt - v) ** 2).sum()
        loss.backward()
        A, Bm = A - eta[0, 0, t] * At.grad.numpy(), Bm - eta[0, 0, t] * Bt.grad.numpy()
        if _rel(Z[0, 0, t], _gelu_t(Q[0, 0, t][None] @ A)[0] @ Bm) > 1e-12:
            return False
    return _rel(A1[0, 0], A) < 1e-12 and _rel(A2[0, 0], Bm) < 1e-12


def pin_backward_finite_differences(M):
    # gradient of L = sum(dZ . Z) + sum(dWT . W_T), Z and W_T from the token-level definition
    rng = np.random.default_rng(10)
    Q, K, V, eta, W0 = _lin(1, 1, 5, 3, 10)
    dZ, dWT = rng.standard_normal(Q.shape), rng.standard_normal(W0.shape)
    for chunk in (2, 5):
        g = M.linear_backward(Q, K, V, eta, W0, dZ, dWT, chunk)
        args = [Q, K, V, eta, W0]

        def L(*a):
            Z, W = M.linear_primal(*a, chunk)
            return float(np.sum(dZ * Z) + np.sum(dWT * W))

        for ai, a in enumerate(args):
            fd = np.zeros_like(a)
            for idx in np.ndindex(a.shape):
                ap = [x.copy() for x in args]
                am = [x.copy() for x in args]
                ap[ai][idx] += 1e-5
                am[ai][idx] -= 1e-5
                fd[idx] = (L(*ap) - L(*am)) / 2e-5
            if np.max(np.abs(g[ai] - fd)) > 1e-7 * max(1.0, np.max(np.abs(fd))):
                return False
    return True


def pin_mlp_backward_finite_differences(M):
    # gradient of L = sum(dZ . Z) + sum(dW1T . W1_T) + sum(dW2T . W2_T) of the token-level TTT-MLP scan
    rng = np.random.default_rng(11)
    Q, K, V, eta, W1, W2 = _mlp(1, 1, 4, 2, 3, 11)
    dZ, dW1T, dW2T = rng.standard_normal(Q.shape), rng.standard_normal(W1.shape), rng.standard_normal(W2.shape)
    args = [Q, K, V, eta, W1, W2]
    for chunk in (3,):
        g = M.mlp_backward(Q, K, V, eta, W1, W2, dZ, dW1T, dW2T, chunk)

        def L(*a):
            Z, A, Bm = M.mlp_primal(*a, chunk)
            return float(np.sum(dZ * Z) + np.sum(dW1T * A) + np.sum(dW2T * Bm))

        for ai, a in enumerate(args):
            fd = np.zeros_like(a)
            for idx in np.ndindex(a.shape):
                ap = [x.copy() for x in args]
                am = [x.copy() for x in args]
                ap[ai][idx] += 1e-5
                am[ai][idx] -= 1e-5
                fd[idx] = (L(*ap) - L(*am)) / 2e-5
            if np.max(np.abs(g[ai] - fd)) > 2e-7 * max(1.0, np.max(np.abs(fd))):
                return False
    return True


def pin_gelu_second(M):
    h = 1e-5
    return all(abs(M.gelu_second(x) - (M.gelu_prime(x + h) - M.gelu_prime(x - h)) / (2 * h)) < 1e-8
               for x in (-2.3, -0.4, 0.0, 0.7, 3.1))


def pin_momentum(M):
    # beta = 0 is the plain scan; primal = closed form; chunk 1 is heavy-ball SGD (torch autograd)
    Q, K, V, eta, W0 = _lin(1, 2, 13, 4, 12)
    M0 = np.random.default_rng(12).standard_normal(W0.shape) * 0.2
    Zr, Wr = M.linear_primal(Q, K, V, eta, W0, 3)
    for fn in (M.linear_momentum_primal, M.linear_momentum_dual):
        Z, W, _ = fn(Q, K, V, eta, W0, M0, 0.0, 3)
        if _rel(Z, Zr) > 1e-12 or _rel(W, Wr) > 1e-12:
            return False
    a = M.linear_momentum_primal(Q, K, V, eta, W0, M0, 0.6, 3)
    b = M.linear_momentum_dual(Q, K, V, eta, W0, M0, 0.6, 3)
    if any(_rel(y, x) > 1e-12 for x, y in zip(a, b)):
        return False
    Z, W, Mo = M.linear_momentum_primal(Q, K, V, eta, W0, M0, 0.6, 1)
    Wt, Mt = torch.tensor(W0[0, 0]), torch.tensor(M0[0, 0])
    for t in range(13):
        w = Wt.clone().requires_grad_(True)
        (0.5 * ((torch.tensor(K[0, 0, t]) @ w - torch.tensor(V[0, 0, t])) ** 2).sum()).backward()
        Mt = 0.6 * Mt + w.grad
        Wt = Wt - eta[0, 0, t] * Mt
        if _rel(Z[0, 0, t], (torch.tensor(Q[0, 0, t]) @ Wt).numpy()) > 1e-12:
            return False
    return _rel(W[0, 0], Wt.numpy()) < 1e-12 and _rel(Mo[0, 0], Mt.numpy()) < 1e-12


PINS = [pin_golden, pin_primal_dual, pin_linear_attention, pin_delta_rule, pin_consistent_targets,
        pin_mlp_kernelised_attention, pin_mlp_finite_differences, pin_gelu, pin_mlp_online_gd,
        pin_backward_finite_differences, pin_mlp_backward_finite_differences, pin_gelu_second, pin_momentum]


def _bind(src_text, tmpdir, tag):
    """Fresh instance of the oracle binding over a compiled copy of `src_text`."""
    csrc = os.path.join(tmpdir, f"ttt_oracle_{tag}.c")
    with open(csrc, "w") as f:
        f.write(src_text)
    spec = importlib.util.spec_from_file_location(f"oracle_{tag}", BINDING)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = csrc
    mod._LIB = os.path.join(tmpdir, f"_ttt_oracle_{tag}.so")
    mod._lib = None
    mod.build(force=True)
    return mod


def _failed_pins(M):
    out = []
    for p in PINS:
        try:
            ok = p(M)
        except (AssertionError, FloatingPointError, ValueError):
            ok = False
        if not ok:
            out.append(p.__name__)
    return out


def test_every_pin_passes_on_the_oracle(tmp_path):
    M = _bind(open(SRC).read(), str(tmp_path), "orig")
    assert _failed_pins(M) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not unique or missing: {name}"
    M = _bind(src.replace(old, new), str(tmp_path), "mut")
    assert _failed_pins(M), f"no pin catches the mutant: {name}"
