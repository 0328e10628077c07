"""GPU parity of the TTT-Linear prefill with momentum (ttt_linear_momentum_prefill) against the fp64
oracle, through the C ABI: Z, the final fast weights and the final momentum.

Error metric max|delta| / ||ref||_inf per output; bar 1e-4 for fp32 inputs and 2e-2 for bf16.
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


def _m0(x, seed, zero=False):
    if zero:
        return None
    rng = np.random.default_rng(seed)
    return WL.round_to(rng.standard_normal(tuple(x["W0"].shape)) * 0.02, "f32")


CASES = [(200, 16), (200, 37), (64, 1), (96, 64), (300, 512), (13, 16)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 64, 128])
@pytest.mark.parametrize("T_,chunk", CASES)
@pytest.mark.parametrize("beta", [0.0, 0.5, 0.9])
def test_momentum_small_shapes(dtype, d, T_, chunk, beta):
    x = WL.linear_inputs(2, 3, T_, d, seed=3000 + d + T_ + chunk, dtype=dtype)
    M0 = _m0(x, 3100 + d, zero=(chunk == 37))
    g = cuda(x)
    Z, W, M = T.linear_momentum_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W0"],
                                        None if M0 is None else M0.cuda(), chunk, beta)
    torch.cuda.synchronize()
    r = f64(x)
    Zr, Wr, Mr = O.linear_momentum_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"],
                                        None if M0 is None else WL.to_f64(M0), beta, chunk)
    assert rel_err(Z, Zr) <= TOL[dtype]
    assert rel_err(W, Wr) <= TOL[dtype]
    assert rel_err(M, Mr) <= TOL[dtype]


def test_momentum_zero_beta_matches_the_plain_prefill():
    x = WL.linear_inputs(2, 2, 96, 32, seed=3200, dtype="f32")
    g = cuda(x)
    Z, W, _ = T.linear_momentum_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W0"], None, 16, 0.0)
    Z1, W1 = T.linear_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W0"], 16)
    torch.cuda.synchronize()
    assert torch.allclose(Z, Z1, rtol=1e-5, atol=1e-6) and torch.allclose(W, W1, rtol=1e-5, atol=1e-6)


def test_momentum_in_place_split_and_resume():
    # two calls chained through (W, M) at a block boundary, both updated in place, equal one pass
    x = WL.linear_inputs(2, 2, 128, 64, seed=3300, dtype="bf16")
    M0 = _m0(x, 3301)
    g = cuda(x)
    W, M = g["W0"].clone(), M0.cuda()
    parts = []
    for lo, hi in ((0, 48), (48, 128)):
        sl = lambda t: t[:, :, lo:hi].contiguous()
        Zp = torch.empty_like(sl(g["Q"]))
        T.ttt_linear_momentum_prefill(sl(g["Q"]), sl(g["K"]), sl(g["V"]), sl(g["eta"]), W, M, Zp, W, M, 16, 0.9)
        parts.append(Zp)
    torch.cuda.synchronize()
    r = f64(x)
    Zr, Wr, Mr = O.linear_momentum_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], WL.to_f64(M0), 0.9, 16)
    assert rel_err(torch.cat(parts, 2), Zr) <= TOL["bf16"]
    assert rel_err(W, Wr) <= TOL["bf16"] and rel_err(M, Mr) <= TOL["bf16"]


def test_momentum_empty_sequence_passes_the_state_through():
    x = cuda(WL.linear_inputs(1, 2, 16, 32, seed=3400, dtype="f32"))
    e = torch.empty(1, 2, 0, 32, device="cuda")
    Wo, Mo = torch.full_like(x["W0"], 7.0), torch.full_like(x["W0"], 7.0)
    T.ttt_linear_momentum_prefill(e, e, e, torch.empty(1, 2, 0, device="cuda"), x["W0"], None, e, Wo, Mo, 16, 0.5)
    torch.cuda.synchronize()
    assert torch.equal(Wo, x["W0"]) and torch.count_nonzero(Mo) == 0


def test_momentum_headline_shape_all_heads():
    # B=8 H=12 d=64 T=2048 chunk=16 bf16, beta = 0.9: every element of all 96 sequences
    w = WL.WORKLOADS["linear_prefill"]
    x = WL.workload_inputs(w)
    M0 = _m0(x, 3500)
    g = cuda(x)
    Z, W, M = T.linear_momentum_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W0"], M0.cuda(), w.chunk, 0.9)
    torch.cuda.synchronize()
    r = f64(x)
    Zr, Wr, Mr = O.linear_momentum_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], WL.to_f64(M0), 0.9, w.chunk)
    check("linear_momentum B=8 H=12 d=64 T=2048 b=16 beta=0.9", TOL["bf16"], Z=(Z, Zr), W=(W, Wr), M=(M, Mr))


# bf16, d = 64, chunk 16 runs the warp-MMA kernel; T = 157 / 7 / 1001 end in a partial chunk (its
# momentum decays by beta per token it holds, not per 16), 1001 with several stages
@pytest.mark.parametrize("beta", [0.0, 0.5, 0.9, 1.0])
@pytest.mark.parametrize("B,H", [(2, 3), (1, 1)])  # 6 heads: one CTA per head; 1 head: one per column group
@pytest.mark.parametrize("T_", [160, 157, 7, 1001])
def test_momentum_mma_shape(beta, B, H, T_):
    x = WL.linear_inputs(B, H, T_, 64, seed=3600 + B * H + T_, dtype="bf16")
    M0 = _m0(x, 3601, zero=(beta == 0.5))
    g = cuda(x)
    Z, W, M = T.linear_momentum_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W0"],
                                        None if M0 is None else M0.cuda(), 16, beta)
    torch.cuda.synchronize()
    r = f64(x)
    Zr, Wr, Mr = O.linear_momentum_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"],
                                        None if M0 is None else WL.to_f64(M0), beta, 16)
    assert rel_err(Z, Zr) <= TOL["bf16"]
    assert rel_err(W, Wr) <= TOL["bf16"]
    assert rel_err(M, Mr) <= TOL["bf16"]


def test_momentum_mma_and_simt_kernels_agree(monkeypatch):
    x = WL.linear_inputs(2, 2, 256, 64, seed=3700, dtype="bf16")
    M0 = _m0(x, 3701)
    g = cuda(x)
    a = T.linear_momentum_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W0"], M0.cuda(), 16, 0.9)
    monkeypatch.setenv("TTT_LINEAR_MOMENTUM_KERNEL", "simt")
    b = T.linear_momentum_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W0"], M0.cuda(), 16, 0.9)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert rel_err(u, v.double().cpu().numpy()) <= TOL["bf16"]


@pytest.mark.parametrize("B,H", [(4, 12), (4, 75)])  # two column groups per CTA; four, more CTAs than SMs
def test_momentum_mma_column_group_layouts(B, H):
    x = WL.linear_inputs(B, H, 96, 64, seed=3800 + H, dtype="bf16")
    M0 = _m0(x, 3801 + H)
    g = cuda(x)
    Z, W, M = T.linear_momentum_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W0"], M0.cuda(), 16, 0.8)
    torch.cuda.synchronize()
    r = f64(x)
    Zr, Wr, Mr = O.linear_momentum_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], WL.to_f64(M0), 0.8, 16)
    assert rel_err(Z, Zr) <= TOL["bf16"]
    assert rel_err(W, Wr) <= TOL["bf16"]
    assert rel_err(M, Mr) <= TOL["bf16"]
