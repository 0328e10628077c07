"""GPU parity of the TTT-Linear backward (and of the forward that records the block-start
states) against the fp64 oracle, through the C ABI.

Error metric: max|delta| / ||ref||_inf per output (dQ, dK, dV, deta, dW0 and the recorded
states); bar 1e-4 for fp32 inputs and 2e-2 for bf16 inputs.  The incoming gradients dZ and
dW_T are seeded draws (workloads.backward_inputs); the oracle reads the same rounded values.
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


def _run(x, g, chunk):
    xc = cuda(x)
    Z, W, Wh = T.linear_prefill_hist(xc["Q"], xc["K"], xc["V"], xc["eta"], xc["W0"], chunk)
    dWT = g["dWT"].cuda() if g["dWT"] is not None else None
    grads = T.linear_prefill_backward(xc["Q"], xc["K"], xc["V"], xc["eta"], Wh, g["dZ"].cuda(), dWT, chunk)
    torch.cuda.synchronize()
    return Z, W, Wh, grads


def _oracle(x, g, chunk):
    r = f64(x)
    dWT = WL.to_f64(g["dWT"]) if g["dWT"] is not None else None
    return O.linear_backward(r["Q"], r["K"], r["V"], r["eta"], r["W0"], WL.to_f64(g["dZ"]), dWT, chunk)


CASES = [  # B, H, T, d, chunk, dtype, with dW_T
    (2, 3, 64, 16, 16, "f32", True),
    (1, 2, 50, 32, 8, "f32", True),      # short last block
    (2, 1, 37, 64, 1, "f32", False),     # online steps
    (1, 2, 100, 64, 64, "f32", True),    # short last block of a long chunk
    (2, 2, 128, 64, 16, "bf16", True),
    (1, 2, 96, 64, 32, "bf16", False),
    (1, 2, 48, 128, 16, "bf16", True),
    (1, 1, 20, 128, 3, "f32", True),
]


@pytest.mark.parametrize("B,H,T_,d,chunk,dtype,with_dWT", CASES)
def test_backward_matches_oracle(B, H, T_, d, chunk, dtype, with_dWT):
    x = WL.linear_inputs(B, H, T_, d, seed=700 + T_ + d + chunk, dtype=dtype, w_std=0.05)
    g = WL.backward_inputs(B, H, T_, d, seed=800 + T_ + d + chunk, dtype=dtype, with_dWT=with_dWT)
    Z, W, Wh, grads = _run(x, g, chunk)
    r = f64(x)
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], chunk)
    assert rel_err(Z, Zr) <= TOL[dtype] and rel_err(W, Wr) <= TOL[dtype]
    ref = _oracle(x, g, chunk)
    for name, got, want in zip(("dQ", "dK", "dV", "deta", "dW0"), grads, ref):
        assert rel_err(got, want) <= TOL[dtype], name


@pytest.mark.parametrize("kernel", ["mma", "simt"])
@pytest.mark.parametrize("B,H,T_,with_dWT", [(1, 1, 16, True), (2, 3, 48, False), (1, 2, 208, True),
                                             (4, 40, 64, True), (1, 2, 1040, False), (2, 3, 1037, True),
                                             (1, 2, 1036, False), (2, 1, 7, True), (1, 3, 67, True)])
def test_backward_kernels_d64_blocks_of_16(kernel, B, H, T_, with_dWT, monkeypatch):
    # bf16, d = 64, blocks of 16: the tensor-core backward (default) and the SIMT one; stages of
    # four blocks with and without a short last stage, more CTAs than SMs, and T not a multiple of
    # 16 (a partial last block, the first processed; with 4 not dividing T every eta by cp.async)
    if kernel == "simt":
        monkeypatch.setenv("TTT_LINEAR_BACKWARD_KERNEL", "simt")
    else:
        monkeypatch.delenv("TTT_LINEAR_BACKWARD_KERNEL", raising=False)
    x = WL.linear_inputs(B, H, T_, 64, seed=1100 + T_ + H, dtype="bf16", w_std=0.05)
    g = WL.backward_inputs(B, H, T_, 64, seed=1200 + T_ + H, dtype="bf16", with_dWT=with_dWT)
    _, _, _, grads = _run(x, g, 16)
    ref = _oracle(x, g, 16)
    for name, got, want in zip(("dQ", "dK", "dV", "deta", "dW0"), grads, ref):
        assert rel_err(got, want) <= TOL["bf16"], name


def test_recorded_states_are_the_block_start_states():
    # W_hist[n] is the state after the first n blocks: the final state of a prefill over them
    x = WL.linear_inputs(2, 2, 80, 32, seed=901, dtype="f32", w_std=0.05)
    _, W, Wh, _ = _run(x, WL.backward_inputs(2, 2, 80, 32, seed=902, dtype="f32"), 16)
    r = f64(x)
    assert Wh.shape == (2, 2, 5, 32, 32)
    assert torch.equal(Wh[:, :, 0], x["W0"].cuda())
    for n in range(1, 5):
        cut = {k: (v[:, :, :16 * n] if k != "W0" else v) for k, v in r.items()}
        _, Wn = O.linear_dual(cut["Q"], cut["K"], cut["V"], cut["eta"], cut["W0"], 16)
        assert rel_err(Wh[:, :, n], Wn) <= TOL["f32"]


@pytest.mark.parametrize("d", [64, 128])
def test_recorded_states_tensor_core_forward(d):
    # bf16, blocks of 16: the warp-MMA forward records the states; compare with prefixes in the oracle
    x = WL.linear_inputs(1, 3, 96, d, seed=905 + d, dtype="bf16", w_std=0.05)
    g = WL.backward_inputs(1, 3, 96, d, seed=906, dtype="bf16")
    Z, W, Wh, _ = _run(x, g, 16)
    r = f64(x)
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], 16)
    assert rel_err(Z, Zr) <= TOL["bf16"] and rel_err(W, Wr) <= TOL["bf16"]
    # bf16 runs record the states rounded to bf16 (round to nearest even)
    assert Wh.dtype == torch.bfloat16 and torch.equal(Wh[:, :, 0], x["W0"].cuda().to(torch.bfloat16))
    for n in (1, 2, 5):
        cut = {k: (v[:, :, :16 * n] if k != "W0" else v) for k, v in r.items()}
        _, Wn = O.linear_dual(cut["Q"], cut["K"], cut["V"], cut["eta"], cut["W0"], 16)
        assert rel_err(Wh[:, :, n], Wn) <= TOL["bf16"]


def test_backward_headline_shape_all_heads():
    # B=8 H=12 d=64 T=2048 chunk=16 bf16: every element of dQ, dK, dV, deta and dW0 of all 96
    # sequences, and the recording forward's Z and final state, against the oracle
    w = WL.WORKLOADS["linear_prefill"]
    x = WL.workload_inputs(w)
    g = WL.backward_inputs(w.B, w.H, w.T, w.d, seed=w.seed + 100, dtype=w.dtype)
    Z, W, _, grads = _run(x, g, w.chunk)
    r = f64(x)
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], w.chunk)
    ref = _oracle(x, g, w.chunk)
    check("linear_backward B=8 H=12 d=64 T=2048 b=16 (recording forward, gradients)", TOL["bf16"],
          Z=(Z, Zr), W=(W, Wr), **{n: (got, want) for n, got, want in
                                   zip(("dQ", "dK", "dV", "deta", "dW0"), grads, ref)})


def test_backward_without_tokens_passes_the_state_gradient_through():
    dWT = torch.randn(1, 2, 16, 16, device="cuda")
    dW0 = torch.full_like(dWT, 3.0)
    e = torch.empty(1, 2, 0, 16, device="cuda")
    Wh = torch.empty(1, 2, 0, 16, 16, device="cuda")
    de = torch.empty(1, 2, 0, device="cuda")
    T.ttt_linear_prefill_backward(e, e, e, de, Wh, e, dWT, e, e, e, de, dW0, 16)
    torch.cuda.synchronize()
    assert torch.equal(dW0, dWT)
    T.ttt_linear_prefill_backward(e, e, e, de, Wh, e, None, e, e, e, de, dW0, 16)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dW0) == 0


def test_backward_deterministic():
    x = WL.linear_inputs(2, 2, 64, 64, seed=903, dtype="bf16")
    g = WL.backward_inputs(2, 2, 64, 64, seed=904, dtype="bf16")
    a = _run(x, g, 16)[3]
    b = _run(x, g, 16)[3]
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_recorded_states_headline_all_heads():
    # B=8 H=12 d=64 T=2048 b=16 bf16: the recording forward (one-pass kernel, four column groups per CTA,
    # states written by TMA stores) against the oracle's state after n blocks, every head
    w = WL.WORKLOADS["linear_prefill"]
    x = WL.workload_inputs(w)
    xc = cuda(x)
    Z, W, Wh = T.linear_prefill_hist(xc["Q"], xc["K"], xc["V"], xc["eta"], xc["W0"], w.chunk)
    torch.cuda.synchronize()
    assert torch.equal(Wh[:, :, 0], xc["W0"].to(torch.bfloat16))
    r = f64(x)
    for n in (1, 37, 127):
        cut = {k: (v[:, :, :16 * n] if k != "W0" else v) for k, v in r.items()}
        _, Wn = O.linear_dual(cut["Q"], cut["K"], cut["V"], cut["eta"], cut["W0"], 16)
        assert rel_err(Wh[:, :, n], Wn) <= TOL["bf16"], n


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T_", [23, 205])
def test_recorded_states_partial_last_sub_block(d, T_):
    # bf16, chunk 16, T not a multiple of 16: the tensor-core forward records ceil(T / 16) states;
    # the gradients through them (SIMT backward) match the oracle
    x = WL.linear_inputs(2, 2, T_, d, seed=930 + T_ + d, dtype="bf16", w_std=0.05)
    g = WL.backward_inputs(2, 2, T_, d, seed=931 + T_ + d, dtype="bf16")
    Z, W, Wh, grads = _run(x, g, 16)
    r = f64(x)
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], 16)
    assert Wh.shape == (2, 2, (T_ + 15) // 16, d, d)
    assert rel_err(Z, Zr) <= TOL["bf16"] and rel_err(W, Wr) <= TOL["bf16"]
    for n in range(1, Wh.shape[2]):
        cut = {k: (v[:, :, :16 * n] if k != "W0" else v) for k, v in r.items()}
        _, Wn = O.linear_dual(cut["Q"], cut["K"], cut["V"], cut["eta"], cut["W0"], 16)
        assert rel_err(Wh[:, :, n], Wn) <= TOL["bf16"]
    for got, want in zip(grads, _oracle(x, g, 16)):
        assert rel_err(got, want) <= TOL["bf16"]
