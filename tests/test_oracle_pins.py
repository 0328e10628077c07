"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

* exact hand-derived d=2 examples (tests/golden/linear_d2_hand.json);
* closed forms: causal linear attention when W0 = 0 (the TTT essay's
  linear-attention remark), the delta rule for one-token blocks, the kernelised
  linear attention that TTT-MLP reduces to when W2 = 0;
* invariants: eta = 0, V = f(K; W0), joint linearity, column permutation,
  split-and-chain at a block boundary;
* the MLP gradient against central finite differences, GELU against torch's
  tanh-form GELU and GELU' against autograd;
* the token-level (primal) and matrix (dual) evaluations against each other.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O
from test_sequence_layers_07_b300 import workloads as WL

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _rand_linear(B, H, T, d, seed, eta_scale=None, w_std=0.3):
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((B, H, T, d)) / math.sqrt(d)
    K = rng.standard_normal((B, H, T, d)) / math.sqrt(d)
    V = rng.standard_normal((B, H, T, d)) / math.sqrt(d)
    eta = rng.uniform(0.05, 0.6, (B, H, T)) if eta_scale is None else np.full((B, H, T), eta_scale)
    W0 = rng.standard_normal((B, H, d, d)) * w_std
    return Q, K, V, eta, W0


def _rand_mlp(B, H, T, d, hd, seed, w_std=0.5):
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((B, H, T, d)) / math.sqrt(d)
    K = rng.standard_normal((B, H, T, d)) / math.sqrt(d)
    V = rng.standard_normal((B, H, T, d)) / math.sqrt(d)
    eta = rng.uniform(0.05, 0.5, (B, H, T))
    W1 = rng.standard_normal((B, H, d, hd)) * w_std
    W2 = rng.standard_normal((B, H, hd, d)) * w_std
    return Q, K, V, eta, W1, W2


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ---------------------------------------------------------------- golden d=2

@pytest.mark.parametrize("fn", ["primal", "dual"])
def test_hand_examples_d2(golden_dir, fn):
    g = json.load(open(os.path.join(golden_dir, "linear_d2_hand.json")))
    inp = g["inputs"]
    q = np.array(inp["q"], float)[None, None]
    k = np.array(inp["k"], float)[None, None]
    v = np.array(inp["v"], float)[None, None]
    for case in g["cases"]:
        W0 = np.array(inp["W0"], float) if case["W0"] == "inputs" else np.zeros((2, 2))
        eta = np.array(case["eta"], float)[None, None]
        f = O.linear_primal if fn == "primal" else O.linear_dual
        Z, W = f(q, k, v, eta, W0[None, None], case["chunk"])
        np.testing.assert_allclose(Z[0, 0], np.array(case["Z"]), rtol=0, atol=1e-15, err_msg=case["name"])
        np.testing.assert_allclose(W[0, 0], np.array(case["W"]), rtol=0, atol=1e-15, err_msg=case["name"])


def test_decode_matches_hand_online_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "linear_d2_hand.json")))
    case = [c for c in g["cases"] if c["chunk"] == 1][0]
    W = np.array(g["inputs"]["W0"], float)[None, None]
    for t in range(2):
        q = np.array(g["inputs"]["q"][t], float)[None, None]
        k = np.array(g["inputs"]["k"][t], float)[None, None]
        v = np.array(g["inputs"]["v"][t], float)[None, None]
        z, W = O.linear_decode(q, k, v, np.array([[case["eta"][t]]]), W)
        np.testing.assert_allclose(z[0, 0], case["Z"][t], atol=1e-15)
    np.testing.assert_allclose(W[0, 0], case["W"], atol=1e-15)


# ------------------------------------------------------------ primal vs dual

@pytest.mark.parametrize("chunk", [1, 2, 5, 16, 64])
def test_linear_primal_equals_dual(chunk):
    Q, K, V, eta, W0 = _rand_linear(2, 3, 70, 8, seed=chunk)  # 70: ragged last block for 16, 64
    Zp, Wp = O.linear_primal(Q, K, V, eta, W0, chunk)
    Zd, Wd = O.linear_dual(Q, K, V, eta, W0, chunk)
    assert _rel(Zd, Zp) < 1e-12 and _rel(Wd, Wp) < 1e-12


@pytest.mark.parametrize("chunk", [1, 3, 16])
def test_mlp_primal_equals_dual(chunk):
    Q, K, V, eta, W1, W2 = _rand_mlp(1, 2, 37, 6, 12, seed=10 + chunk)
    Zp, W1p, W2p = O.mlp_primal(Q, K, V, eta, W1, W2, chunk)
    Zd, W1d, W2d = O.mlp_dual(Q, K, V, eta, W1, W2, chunk)
    assert _rel(Zd, Zp) < 1e-12 and _rel(W1d, W1p) < 1e-12 and _rel(W2d, W2p) < 1e-12


# ------------------------------------------------------------- closed forms

@pytest.mark.parametrize("fn", [O.linear_primal, O.linear_dual])
def test_zero_init_whole_sequence_is_causal_linear_attention(fn):
    # linear inner model, zero initial state, one block: z_i = sum_{j<=i} eta_j (q_i.k_j) v_j
    Q, K, V, eta, _ = _rand_linear(1, 2, 24, 5, seed=3)
    W0 = np.zeros((1, 2, 5, 5))
    Z, W = fn(Q, K, V, eta, W0, 24)
    for h in range(2):
        S = Q[0, h] @ K[0, h].T
        Zla = np.zeros((24, 5))
        for i in range(24):
            for j in range(i + 1):
                Zla[i] += eta[0, h, j] * S[i, j] * V[0, h, j]
        WT = sum(eta[0, h, j] * np.outer(K[0, h, j], V[0, h, j]) for j in range(24))
        assert _rel(Z[0, h], Zla) < 1e-13
        assert _rel(W[0, h], WT) < 1e-13


def test_zero_init_first_block_is_linear_attention_even_with_more_blocks():
    Q, K, V, eta, _ = _rand_linear(1, 1, 32, 4, seed=4)
    Z, _ = O.linear_dual(Q, K, V, eta, np.zeros((1, 1, 4, 4)), 8)
    S = Q[0, 0, :8] @ K[0, 0, :8].T
    Zla = np.array([sum(eta[0, 0, j] * S[i, j] * V[0, 0, j] for j in range(i + 1)) for i in range(8)])
    assert _rel(Z[0, 0, :8], Zla) < 1e-13


@pytest.mark.parametrize("fn", [O.linear_primal, O.linear_dual])
def test_online_blocks_follow_delta_rule(fn):
    # textbook delta rule: W_t = (I - eta_t k_t^T k_t) W_{t-1} + eta_t k_t^T v_t, z_t = q_t W_t
    Q, K, V, eta, W0 = _rand_linear(1, 1, 20, 6, seed=5)
    Z, W = fn(Q, K, V, eta, W0, 1)
    Wt = W0[0, 0].copy()
    for t in range(20):
        k, v = K[0, 0, t], V[0, 0, t]
        Wt = (np.eye(6) - eta[0, 0, t] * np.outer(k, k)) @ Wt + eta[0, 0, t] * np.outer(k, v)
        assert _rel(Z[0, 0, t], Q[0, 0, t] @ Wt) < 1e-12
    assert _rel(W[0, 0], Wt) < 1e-12


def test_block_step_is_affine_map_of_the_block_start_state():
    # one block of b tokens with gradients at W_s: W' = (I - K^T D K) W_s + K^T D V
    Q, K, V, eta, W0 = _rand_linear(1, 1, 12, 5, seed=6)
    _, W = O.linear_primal(Q, K, V, eta, W0, 12)
    Kc, Vc, D = K[0, 0], V[0, 0], np.diag(eta[0, 0])
    Wexp = (np.eye(5) - Kc.T @ D @ Kc) @ W0[0, 0] + Kc.T @ D @ Vc
    assert _rel(W[0, 0], Wexp) < 1e-13


def test_mlp_zero_second_layer_is_kernelised_linear_attention():
    # W2 = 0: first block leaves W1 unchanged; z_i = sum_{j<=i} eta_j (hq_i.hk_j) v_j with
    # hq = GELU(q W1), hk = GELU(k W1); W2 = Hk^T diag(eta) V
    Q, K, V, eta, W1, _ = _rand_mlp(1, 1, 9, 4, 7, seed=7)
    W2 = np.zeros((1, 1, 7, 4))
    gelu_t = lambda x: torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    for fn in (O.mlp_primal, O.mlp_dual):
        Z, W1o, W2o = fn(Q, K, V, eta, W1, W2, 9)
        Hq, Hk = gelu_t(Q[0, 0] @ W1[0, 0]), gelu_t(K[0, 0] @ W1[0, 0])
        Zexp = np.array([sum(eta[0, 0, j] * (Hq[i] @ Hk[j]) * V[0, 0, j] for j in range(i + 1))
                         for i in range(9)])
        assert _rel(Z[0, 0], Zexp) < 1e-12
        assert _rel(W1o, W1) < 1e-15
        assert _rel(W2o[0, 0], Hk.T @ np.diag(eta[0, 0]) @ V[0, 0]) < 1e-12


# --------------------------------------------------------------- invariants

def test_linear_zero_eta_is_plain_readout():
    Q, K, V, _, W0 = _rand_linear(2, 2, 33, 7, seed=8)
    Z, W = O.linear_dual(Q, K, V, np.zeros((2, 2, 33)), W0, 16)
    assert _rel(Z, Q @ W0) < 1e-14 and np.array_equal(W, W0)


def test_linear_consistent_targets_leave_state_unchanged():
    Q, K, _, eta, W0 = _rand_linear(1, 2, 40, 6, seed=9)
    V = K @ W0
    for fn in (O.linear_primal, O.linear_dual):
        Z, W = fn(Q, K, V, eta, W0, 8)
        assert _rel(W, W0) < 1e-14 and _rel(Z, Q @ W0) < 1e-14


def test_mlp_zero_eta_and_consistent_targets():
    Q, K, V, eta, W1, W2 = _rand_mlp(1, 2, 20, 5, 9, seed=11)
    gelu_t = lambda x: torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    Z, W1o, W2o = O.mlp_dual(Q, K, V, np.zeros_like(eta), W1, W2, 4)
    assert _rel(Z, gelu_t(Q @ W1) @ W2) < 1e-13 and np.array_equal(W1o, W1) and np.array_equal(W2o, W2)
    V2 = gelu_t(K @ W1) @ W2
    for fn in (O.mlp_primal, O.mlp_dual):
        Z, W1o, W2o = fn(Q, K, V2, eta, W1, W2, 4)
        assert _rel(W1o, W1) < 1e-13 and _rel(W2o, W2) < 1e-13
        assert _rel(Z, gelu_t(Q @ W1) @ W2) < 1e-12


def test_linear_jointly_linear_in_state_and_targets():
    Q, K, V, eta, W0 = _rand_linear(1, 1, 24, 6, seed=12)
    Z1, W1 = O.linear_dual(Q, K, V, eta, W0, 8)
    Z2, W2 = O.linear_dual(Q, K, -2.5 * V, eta, -2.5 * W0, 8)
    assert _rel(Z2, -2.5 * Z1) < 1e-13 and _rel(W2, -2.5 * W1) < 1e-13


def test_linear_output_column_permutation_equivariance():
    Q, K, V, eta, W0 = _rand_linear(1, 1, 24, 6, seed=13)
    perm = np.array([3, 0, 5, 1, 4, 2])
    Z1, W1 = O.linear_dual(Q, K, V, eta, W0, 8)
    Z2, W2 = O.linear_dual(Q, K, V[..., perm], eta, W0[..., perm], 8)
    assert _rel(Z2, Z1[..., perm]) < 1e-14 and _rel(W2, W1[..., perm]) < 1e-14


@pytest.mark.parametrize("kind", ["linear", "mlp"])
def test_split_and_chain_at_block_boundary(kind):
    if kind == "linear":
        Q, K, V, eta, W0 = _rand_linear(1, 2, 48, 5, seed=14)
        Z, W = O.linear_dual(Q, K, V, eta, W0, 8)
        Za, Wa = O.linear_dual(Q[:, :, :24], K[:, :, :24], V[:, :, :24], eta[:, :, :24], W0, 8)
        Zb, Wb = O.linear_dual(Q[:, :, 24:], K[:, :, 24:], V[:, :, 24:], eta[:, :, 24:], Wa, 8)
        assert _rel(np.concatenate([Za, Zb], 2), Z) < 1e-14 and _rel(Wb, W) < 1e-14
    else:
        Q, K, V, eta, W1, W2 = _rand_mlp(1, 1, 24, 4, 8, seed=15)
        Z, A1, A2 = O.mlp_dual(Q, K, V, eta, W1, W2, 4)
        Za, B1, B2 = O.mlp_dual(Q[:, :, :12], K[:, :, :12], V[:, :, :12], eta[:, :, :12], W1, W2, 4)
        Zb, C1, C2 = O.mlp_dual(Q[:, :, 12:], K[:, :, 12:], V[:, :, 12:], eta[:, :, 12:], B1, B2, 4)
        assert _rel(np.concatenate([Za, Zb], 2), Z) < 1e-14
        assert _rel(C1, A1) < 1e-14 and _rel(C2, A2) < 1e-14


def test_heads_are_independent():
    Q, K, V, eta, W0 = _rand_linear(2, 3, 16, 4, seed=16)
    Z, W = O.linear_dual(Q, K, V, eta, W0, 4)
    Z1, W1 = O.linear_dual(Q[1:2, 2:3], K[1:2, 2:3], V[1:2, 2:3], eta[1:2, 2:3], W0[1:2, 2:3], 4)
    assert np.array_equal(Z[1:2, 2:3], Z1) and np.array_equal(W[1:2, 2:3], W1)


def test_mini_batch_differs_from_online():
    # the block size changes the result (gradients at the block start), so a dropped
    # block-start copy would be caught
    Q, K, V, eta, W0 = _rand_linear(1, 1, 16, 4, seed=17)
    Z1, _ = O.linear_primal(Q, K, V, eta, W0, 1)
    Z4, _ = O.linear_primal(Q, K, V, eta, W0, 4)
    assert _rel(Z1, Z4) > 1e-6


# ------------------------------------------------------------ MLP gradient

def test_gelu_matches_torch_tanh_form():
    xs = np.linspace(-6, 6, 97)
    ref = torch.nn.functional.gelu(torch.from_numpy(xs), approximate="tanh").numpy()
    got = np.array([O.gelu(x) for x in xs])
    assert np.max(np.abs(got - ref)) < 1e-14
    assert O.gelu(0.0) == 0.0
    for x in (0.3, 1.7, 4.0):  # GELU(x) - GELU(-x) = x for the tanh form (tanh is odd)
        assert abs(O.gelu(x) - O.gelu(-x) - x) < 1e-15


def test_gelu_prime_matches_autograd():
    xs = torch.linspace(-6, 6, 97, dtype=torch.float64, requires_grad=True)
    torch.nn.functional.gelu(xs, approximate="tanh").sum().backward()
    got = np.array([O.gelu_prime(float(x)) for x in xs.detach()])
    assert np.max(np.abs(got - xs.grad.numpy())) < 1e-14


def test_mlp_gradient_matches_central_differences():
    rng = np.random.default_rng(18)
    d, hd = 5, 11
    k, v = rng.standard_normal(d), rng.standard_normal(d)
    W1, W2 = rng.standard_normal((d, hd)) * 0.5, rng.standard_normal((hd, d)) * 0.5
    _, a, e1, e2 = O.mlp_token_grad(k, v, W1, W2)
    g1, g2 = np.outer(k, e1), np.outer(a, e2)
    h = 1e-6
    loss = lambda A, Bm: O.mlp_token_grad(k, v, A, Bm)[0]
    fd1 = np.zeros_like(W1)
    for i in range(d):
        for m in range(hd):
            P, M = W1.copy(), W1.copy()
            P[i, m] += h
            M[i, m] -= h
            fd1[i, m] = (loss(P, W2) - loss(M, W2)) / (2 * h)
    fd2 = np.zeros_like(W2)
    for m in range(hd):
        for c in range(d):
            P, M = W2.copy(), W2.copy()
            P[m, c] += h
            M[m, c] -= h
            fd2[m, c] = (loss(W1, P) - loss(W1, M)) / (2 * h)
    assert _rel(g1, fd1) < 1e-6 and _rel(g2, fd2) < 1e-6
    # and the loss is the squared error with the factor 1/2
    y = O.mlp_forward(k, W1, W2)
    assert abs(loss(W1, W2) - 0.5 * np.sum((y - v) ** 2)) < 1e-13


def test_mlp_online_is_plain_gradient_descent():
    # chunk = 1: each token takes one GD step with the (finite-difference pinned) gradient
    Q, K, V, eta, W1, W2 = _rand_mlp(1, 1, 6, 4, 8, seed=19)
    Z, W1o, W2o = O.mlp_primal(Q, K, V, eta, W1, W2, 1)
    A, Bm = W1[0, 0].copy(), W2[0, 0].copy()
    for t in range(6):
        _, a, e1, e2 = O.mlp_token_grad(K[0, 0, t], V[0, 0, t], A, Bm)
        A, Bm = A - eta[0, 0, t] * np.outer(K[0, 0, t], e1), Bm - eta[0, 0, t] * np.outer(a, e2)
        assert _rel(Z[0, 0, t], O.mlp_forward(Q[0, 0, t], A, Bm)) < 1e-13
    assert _rel(W1o[0, 0], A) < 1e-13 and _rel(W2o[0, 0], Bm) < 1e-13


def test_mlp_decode_is_one_token_online_step():
    # the decode oracle is the token-level scan on one token: plain gradient descent (autograd)
    rng = np.random.default_rng(20)
    B, H, d, hd = 2, 1, 4, 6
    q, k, v = (rng.standard_normal((B, H, d)) for _ in range(3))
    eta = rng.uniform(0.1, 0.5, (B, H))
    W1, W2 = rng.standard_normal((B, H, d, hd)) * 0.5, rng.standard_normal((B, H, hd, d)) * 0.5
    z, A, Bm = O.mlp_decode(q, k, v, eta, W1, W2)
    gelu_t = lambda x: torch.nn.functional.gelu(x, approximate="tanh")
    for b in range(B):
        At, Bt = torch.tensor(W1[b, 0], requires_grad=True), torch.tensor(W2[b, 0], requires_grad=True)
        loss = 0.5 * ((gelu_t(torch.tensor(k[b, 0]) @ At) @ Bt - torch.tensor(v[b, 0])) ** 2).sum()
        loss.backward()
        A1 = W1[b, 0] - eta[b, 0] * At.grad.numpy()
        B1 = W2[b, 0] - eta[b, 0] * Bt.grad.numpy()
        assert _rel(A[b, 0], A1) < 1e-12 and _rel(Bm[b, 0], B1) < 1e-12
        zr = (gelu_t(torch.tensor(q[b, 0]) @ torch.tensor(A1)) @ torch.tensor(B1)).numpy()
        assert _rel(z[b, 0], zr) < 1e-12


# ------------------------------------------------------------- workloads

def test_workload_inputs_are_seeded_and_rounded():
    a = WL.linear_inputs(1, 2, 32, 16, seed=5)
    b = WL.linear_inputs(1, 2, 32, 16, seed=5)
    for key in a:
        assert torch.equal(a[key], b[key])
    assert a["Q"].dtype == torch.bfloat16 and a["eta"].dtype == torch.float32
    n = a["K"].double().norm(dim=-1)
    assert torch.all((n - 1).abs() < 1e-2)  # unit rows up to bf16 rounding
    assert torch.all(a["eta"] > 0) and torch.all(a["eta"] < 1.0 / 16)
    assert torch.equal(a["W0"][0, 0], a["W0"][0, 0])


def test_oracle_check_workload_recipe():
    w = WL.WORKLOADS["oracle_check"]
    x = WL.workload_inputs(w)
    assert x["Q"].dtype == torch.float32 and torch.all(x["eta"] == torch.tensor(0.1, dtype=torch.float32))
    assert torch.count_nonzero(x["W0"]) == 0
    kn = x["K"].double().norm(dim=-1)
    assert torch.all((kn - 1).abs() < 1e-6)
    qn = x["Q"].double().norm(dim=-1)
    assert torch.any((qn - 1).abs() > 1e-3)  # q rows are not normalised in this workload
