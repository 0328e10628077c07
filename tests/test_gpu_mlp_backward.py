"""GPU parity of the TTT-MLP backward (and of the forward that records the block-start states)
against the fp64 oracle, through the C ABI.

Error metric: max|delta| / ||ref||_inf per output (dQ, dK, dV, deta, dW1, dW2, the recorded states,
Z and the final states); bar 1e-4 for fp32 inputs and 2e-2 for bf16 inputs.  The incoming
gradients dZ, dW1_T, dW2_T are seeded draws; the oracle reads the same rounded values.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from test_sequence_layers_07_b300 import ttt as T
from test_sequence_layers_07_b300 import workloads as WL
from tests._parity import TOL, check, cuda, f64, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    T.load_library()
    yield
    assert T.ttt_get_device_status() == T.TTT_OK


def _grads(B, H, T_, d, hd, seed, dtype, with_state=True):
    rng = np.random.default_rng(seed)
    dZ = WL.round_to(rng.standard_normal((B, H, T_, d)) / np.sqrt(d), dtype)
    if not with_state:
        return dZ, None, None
    dW1 = WL.round_to(rng.standard_normal((B, H, d, hd)) / np.sqrt(d), "f32")
    dW2 = WL.round_to(rng.standard_normal((B, H, hd, d)) / np.sqrt(d), "f32")
    return dZ, dW1, dW2


def _run(x, dZ, dW1, dW2, chunk):
    g = cuda(x)
    Z, W1, W2, H1, H2 = T.mlp_prefill_hist(g["Q"], g["K"], g["V"], g["eta"], g["W1"], g["W2"], chunk)
    grads = T.mlp_prefill_backward(g["Q"], g["K"], g["V"], g["eta"], H1, H2, dZ.cuda(),
                                   None if dW1 is None else dW1.cuda(), None if dW2 is None else dW2.cuda(), chunk)
    torch.cuda.synchronize()
    return Z, W1, W2, H1, H2, grads


def _oracle(x, dZ, dW1, dW2, chunk):
    r = f64(x)
    return O.mlp_backward(r["Q"], r["K"], r["V"], r["eta"], r["W1"], r["W2"], WL.to_f64(dZ),
                          None if dW1 is None else WL.to_f64(dW1), None if dW2 is None else WL.to_f64(dW2), chunk)


NAMES = ("dQ", "dK", "dV", "deta", "dW1", "dW2")
CASES = [  # B, H, T, d, hidden, chunk, dtype, with state gradients
    (2, 2, 37, 16, 64, 4, "f32", True),    # ragged last block
    (1, 3, 24, 32, 128, 1, "f32", False),  # online steps
    (2, 1, 40, 16, 256, 16, "f32", True),
    (1, 2, 64, 64, 256, 16, "bf16", True),  # the warp-MMA forward records the states
    (2, 2, 50, 64, 256, 16, "bf16", False),  # a partial last block: the warp-MMA forward records the states,
                                             # the SIMT backward reads them
    (1, 2, 48, 32, 64, 8, "bf16", True),
]


@pytest.mark.parametrize("B,H,T_,d,hd,chunk,dtype,with_state", CASES)
def test_mlp_backward_matches_oracle(B, H, T_, d, hd, chunk, dtype, with_state):
    x = WL.mlp_inputs(B, H, T_, d, hd, seed=4000 + T_ + d + hd + chunk, dtype=dtype, w_std=0.1)
    dZ, dW1, dW2 = _grads(B, H, T_, d, hd, 4100 + T_, dtype, with_state)
    Z, W1, W2, H1, H2, grads = _run(x, dZ, dW1, dW2, chunk)
    r = f64(x)
    Zr, W1r, W2r = O.mlp_dual(r["Q"], r["K"], r["V"], r["eta"], r["W1"], r["W2"], chunk)
    assert rel_err(Z, Zr) <= TOL[dtype] and rel_err(W1, W1r) <= TOL[dtype] and rel_err(W2, W2r) <= TOL[dtype]
    ref = _oracle(x, dZ, dW1, dW2, chunk)
    for name, got, want in zip(NAMES, grads, ref):
        assert rel_err(got, want) <= TOL[dtype], name


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_mlp_recorded_states_are_the_block_start_states(dtype):
    x = WL.mlp_inputs(1, 2, 48, 64, 256, seed=4200, dtype=dtype, w_std=0.1)
    g = cuda(x)
    _, _, _, H1, H2 = T.mlp_prefill_hist(g["Q"], g["K"], g["V"], g["eta"], g["W1"], g["W2"], 16)
    torch.cuda.synchronize()
    assert H1.dtype == g["Q"].dtype and H1.shape == (1, 2, 3, 64, 256) and H2.shape == (1, 2, 3, 256, 64)
    assert torch.equal(H1[:, :, 0], g["W1"].to(H1.dtype)) and torch.equal(H2[:, :, 0], g["W2"].to(H2.dtype))
    r = f64(x)
    for n in (1, 2):
        cut = {k: (v[:, :, :16 * n] if k not in ("W1", "W2") else v) for k, v in r.items()}
        _, A, Bm = O.mlp_dual(cut["Q"], cut["K"], cut["V"], cut["eta"], cut["W1"], cut["W2"], 16)
        assert rel_err(H1[:, :, n], A) <= TOL[dtype] and rel_err(H2[:, :, n], Bm) <= TOL[dtype]


def test_mlp_recorded_states_partial_last_block():
    # bf16, d = 64, hidden = 256, T = 45: the warp-MMA forward records ceil(45 / 16) = 3 states
    x = WL.mlp_inputs(1, 2, 45, 64, 256, seed=4210, dtype="bf16", w_std=0.1)
    g = cuda(x)
    Z, W1, W2, H1, H2 = T.mlp_prefill_hist(g["Q"], g["K"], g["V"], g["eta"], g["W1"], g["W2"], 16)
    torch.cuda.synchronize()
    assert H1.shape == (1, 2, 3, 64, 256) and H2.shape == (1, 2, 3, 256, 64)
    r = f64(x)
    Zr, W1r, W2r = O.mlp_dual(r["Q"], r["K"], r["V"], r["eta"], r["W1"], r["W2"], 16)
    assert rel_err(Z, Zr) <= TOL["bf16"] and rel_err(W1, W1r) <= TOL["bf16"] and rel_err(W2, W2r) <= TOL["bf16"]
    for n in (1, 2):
        cut = {k: (v[:, :, :16 * n] if k not in ("W1", "W2") else v) for k, v in r.items()}
        _, A, Bm = O.mlp_dual(cut["Q"], cut["K"], cut["V"], cut["eta"], cut["W1"], cut["W2"], 16)
        assert rel_err(H1[:, :, n], A) <= TOL["bf16"] and rel_err(H2[:, :, n], Bm) <= TOL["bf16"]


def test_mlp_backward_without_tokens_passes_the_state_gradient_through():
    d, hd = 16, 64
    dW1 = torch.randn(1, 2, d, hd, device="cuda")
    dW2 = torch.randn(1, 2, hd, d, device="cuda")
    o1, o2 = torch.full_like(dW1, 3.0), torch.full_like(dW2, 3.0)
    e = torch.empty(1, 2, 0, d, device="cuda")
    de = torch.empty(1, 2, 0, device="cuda")
    h1 = torch.empty(1, 2, 0, d, hd, device="cuda")
    h2 = torch.empty(1, 2, 0, hd, d, device="cuda")
    T.ttt_mlp_prefill_backward(e, e, e, de, h1, h2, e, dW1, dW2, e, e, e, de, o1, o2, 16)
    torch.cuda.synchronize()
    assert torch.equal(o1, dW1) and torch.equal(o2, dW2)
    T.ttt_mlp_prefill_backward(e, e, e, de, h1, h2, e, None, None, e, e, e, de, o1, o2, 16)
    torch.cuda.synchronize()
    assert torch.count_nonzero(o1) == 0 and torch.count_nonzero(o2) == 0


def test_mlp_backward_deterministic():
    x = WL.mlp_inputs(1, 3, 64, 64, 256, seed=4300, dtype="bf16", w_std=0.1)
    dZ, dW1, dW2 = _grads(1, 3, 64, 64, 256, 4301, "bf16")
    a = _run(x, dZ, dW1, dW2, 16)[5]
    b = _run(x, dZ, dW1, dW2, 16)[5]
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_mlp_backward_workload_shape_all_heads():
    # the TTT-MLP workload: B=8 H=12 d=64 hidden=256 T=2048 chunk=16 bf16, every element of every
    # gradient of all 96 sequences against the oracle
    w = WL.WORKLOADS["mlp_prefill"]
    x = WL.workload_inputs(w)
    dZ, dW1, dW2 = _grads(w.B, w.H, w.T, w.d, w.hidden, w.seed + 100, w.dtype)
    _, _, _, _, _, grads = _run(x, dZ, dW1, dW2, w.chunk)
    ref = _oracle(x, dZ, dW1, dW2, w.chunk)
    check("mlp_backward B=8 H=12 d=64 h=256 T=2048 b=16", TOL["bf16"],
          **{n: (got, want) for n, got, want in zip(NAMES, grads, ref)})


# bf16, d = 64, hidden = 256, chunk 16 runs the warp-MMA kernel; these cases span several blocks
# and heads of it, and T not a multiple of 16 (a partial last block, the first processed; with 4 not
# dividing T eta comes by 4-byte copies)
@pytest.mark.parametrize("with_state", [True, False])
@pytest.mark.parametrize("T_", [96, 45, 204, 1001])
def test_mlp_backward_mma_shape_matches_oracle(with_state, T_):
    x = WL.mlp_inputs(2, 3, T_, 64, 256, seed=4400 + T_, dtype="bf16", w_std=0.1)
    dZ, dW1, dW2 = _grads(2, 3, T_, 64, 256, 4401 + T_, "bf16", with_state)
    grads = _run(x, dZ, dW1, dW2, 16)[5]
    ref = _oracle(x, dZ, dW1, dW2, 16)
    for name, got, want in zip(NAMES, grads, ref):
        assert rel_err(got, want) <= TOL["bf16"], name


def test_mlp_backward_mma_state_gradient_in_place():
    # dW_T passed as dW_0 (the entry point allows it): read at the start, overwritten with dW_0
    x = WL.mlp_inputs(1, 2, 48, 64, 256, seed=4500, dtype="bf16", w_std=0.1)
    dZ, dW1, dW2 = _grads(1, 2, 48, 64, 256, 4501, "bf16")
    g = cuda(x)
    _, _, _, H1, H2 = T.mlp_prefill_hist(g["Q"], g["K"], g["V"], g["eta"], g["W1"], g["W2"], 16)
    o1, o2 = dW1.cuda(), dW2.cuda()
    dq, dk, dv = (torch.empty_like(g["Q"]) for _ in range(3))
    de = torch.empty_like(g["eta"])
    T.ttt_mlp_prefill_backward(g["Q"], g["K"], g["V"], g["eta"], H1, H2, dZ.cuda(), o1, o2, dq, dk, dv, de, o1, o2, 16)
    torch.cuda.synchronize()
    ref = _oracle(x, dZ, dW1, dW2, 16)
    for name, got, want in zip(NAMES, (dq, dk, dv, de, o1, o2), ref):
        assert rel_err(got, want) <= TOL["bf16"], name


def test_mlp_backward_mma_and_simt_kernels_agree(monkeypatch):
    x = WL.mlp_inputs(2, 2, 64, 64, 256, seed=4600, dtype="bf16", w_std=0.1)
    dZ, dW1, dW2 = _grads(2, 2, 64, 64, 256, 4601, "bf16")
    a = _run(x, dZ, dW1, dW2, 16)[5]
    monkeypatch.setenv("TTT_MLP_BACKWARD_KERNEL", "simt")
    b = _run(x, dZ, dW1, dW2, 16)[5]
    for name, u, v in zip(NAMES, a, b):
        assert rel_err(u, v.double().cpu().numpy()) <= TOL["bf16"], name


def test_mlp_backward_mma_warp_layouts_agree(monkeypatch):
    # eight warps of 32 hidden units (the default) and sixteen of 16 give the same gradients within the bar
    x = WL.mlp_inputs(2, 2, 64, 64, 256, seed=4700, dtype="bf16", w_std=0.1)
    dZ, dW1, dW2 = _grads(2, 2, 64, 64, 256, 4701, "bf16")
    a = _run(x, dZ, dW1, dW2, 16)[5]
    monkeypatch.setenv("TTT_MLP_BACKWARD_WARPS", "16")
    b = _run(x, dZ, dW1, dW2, 16)[5]
    ref = _oracle(x, dZ, dW1, dW2, 16)
    for name, u, v, r in zip(NAMES, a, b, ref):
        assert rel_err(u, r) <= TOL["bf16"] and rel_err(v, r) <= TOL["bf16"], name
        assert rel_err(u, v.double().cpu().numpy()) <= TOL["bf16"], name
