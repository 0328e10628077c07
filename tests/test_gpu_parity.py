"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle.

Error metric: max|delta| / ||ref||_inf per output; bar 1e-4 for fp32 inputs and
2e-2 for bf16 inputs, applied to Z and to every final weight matrix.  Inputs
are the seeded workloads of test_sequence_layers_07_b300.workloads; the oracle
reads exactly the rounded values the GPU reads.
"""
import contextlib
import os

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


def run_linear(x, chunk):
    g = cuda(x)
    Z, W = T.linear_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W0"], chunk)
    torch.cuda.synchronize()
    return Z, W


def run_mlp(x, chunk):
    g = cuda(x)
    Z, W1, W2 = T.mlp_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W1"], g["W2"], chunk)
    torch.cuda.synchronize()
    return Z, W1, W2


# ------------------------------------------------------------------ TTT-Linear

def test_oracle_check_workload_fp32():
    w = WL.WORKLOADS["oracle_check"]
    x = WL.workload_inputs(w)
    Z, W = run_linear(x, w.chunk)
    r = f64(x)
    for fn in (O.linear_dual, O.linear_primal):
        Zr, Wr = fn(r["Q"], r["K"], r["V"], r["eta"], r["W0"], w.chunk)
        assert rel_err(Z, Zr) <= TOL["f32"]
        assert rel_err(W, Wr) <= TOL["f32"]


LIN_CASES = [(200, 16), (200, 37), (64, 1), (96, 64), (300, 512), (13, 16)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("T_,chunk", LIN_CASES)
def test_linear_small_shapes(dtype, d, T_, chunk):
    x = WL.linear_inputs(2, 3, T_, d, seed=100 + d + T_ + chunk, dtype=dtype)
    Z, W = run_linear(x, chunk)
    r = f64(x)
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], chunk)
    assert rel_err(Z, Zr) <= TOL[dtype]
    assert rel_err(W, Wr) <= TOL[dtype]


@contextlib.contextmanager
def linear_kernel(name):
    """Start the TTT-Linear prefill dispatch at kernel `name` ("fused", "tc", "mma" or "generic")."""
    old = os.environ.get("TTT_LINEAR_PREFILL_KERNEL")
    os.environ["TTT_LINEAR_PREFILL_KERNEL"] = name
    try:
        yield
    finally:
        if old is None:
            del os.environ["TTT_LINEAR_PREFILL_KERNEL"]
        else:
            os.environ["TTT_LINEAR_PREFILL_KERNEL"] = old


# d = 64 bf16 shapes the tensor-core kernels take: one 16-token block, stages with and without a
# short last stage, blocks longer than a stage, more CTAs than SMs; B*H = 1..37 runs one column
# group per CTA, 38..74 two, from 75 four (on 148 SMs)
TC_CASES = [(1, 1, 16, 16, 0.02), (2, 3, 128, 16, 0.02), (2, 3, 144, 16, 0.1), (1, 2, 1040, 16, 0.05),
            (2, 2, 256, 32, 0.02), (1, 3, 384, 128, 0.1), (2, 2, 512, 256, 0.02), (1, 2, 1024, 512, 0.05),
            (1, 2, 640, 64, 0.02), (4, 75, 128, 16, 0.02), (2, 24, 272, 16, 0.05), (3, 16, 288, 32, 0.02)]


@pytest.mark.parametrize("kernel", ["fused", "tc", "mma", "generic"])
@pytest.mark.parametrize("B,H,T_,chunk,w_std", TC_CASES)
def test_linear_kernels_d64(kernel, B, H, T_, chunk, w_std):
    x = WL.linear_inputs(B, H, T_, 64, seed=300 + T_ + chunk + H, dtype="bf16", w_std=w_std)
    with linear_kernel(kernel):
        Z, W = run_linear(x, chunk)
    r = f64(x)
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], chunk)
    assert rel_err(Z, Zr) <= TOL["bf16"]
    assert rel_err(W, Wr) <= TOL["bf16"]


def test_linear_prefill_workload_all_heads():
    # B=8 H=12 d=64 T=2048 chunk=16 bf16: every element of Z and of the final state of all 96
    # (batch, head) sequences against the oracle, in the launch configuration the benchmark times
    w = WL.WORKLOADS["linear_prefill"]
    x = WL.workload_inputs(w)
    Z, W = run_linear(x, w.chunk)
    r = f64(x)
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], w.chunk)
    check("linear_prefill B=8 H=12 d=64 T=2048 b=16", TOL["bf16"], Z=(Z, Zr), W=(W, Wr))


@pytest.mark.parametrize("chunk", [16, 64, 512])
def test_long_context_workload_all_heads(chunk):
    # B=1 H=16 d=128 T=32768, bf16: all 16 heads, every element, at each block size of the sweep
    w = WL.WORKLOADS["long_context"]
    x = WL.workload_inputs(w)
    Z, W = run_linear(x, chunk)
    r = f64(x)
    del x
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], chunk)
    check(f"long_context B=1 H=16 d=128 T=32768 b={chunk}", TOL["bf16"], Z=(Z, Zr), W=(W, Wr))


def test_linear_in_place_state_and_split_resume():
    x = WL.linear_inputs(2, 2, 128, 64, seed=7, dtype="bf16")
    g = cuda(x)
    Z_full, W_full = T.linear_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W0"], 16)
    # two calls split at a block boundary, the second resuming from the first's state, in place
    W = g["W0"].clone()
    Za = torch.empty_like(g["Q"][:, :, :48].contiguous())
    T.ttt_linear_prefill(g["Q"][:, :, :48].contiguous(), g["K"][:, :, :48].contiguous(),
                         g["V"][:, :, :48].contiguous(), g["eta"][:, :, :48].contiguous(), W, Za, W, 16)
    Zb = torch.empty_like(g["Q"][:, :, 48:].contiguous())
    T.ttt_linear_prefill(g["Q"][:, :, 48:].contiguous(), g["K"][:, :, 48:].contiguous(),
                         g["V"][:, :, 48:].contiguous(), g["eta"][:, :, 48:].contiguous(), W, Zb, W, 16)
    torch.cuda.synchronize()
    r = f64(x)
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], 16)
    assert rel_err(torch.cat([Za, Zb], 2), Zr) <= TOL["bf16"]
    assert rel_err(W, Wr) <= TOL["bf16"]
    assert rel_err(W_full, Wr) <= TOL["bf16"]


def test_linear_empty_sequence_copies_state():
    x = cuda(WL.linear_inputs(1, 2, 16, 32, seed=3, dtype="f32"))
    Wo = torch.full_like(x["W0"], 7.0)
    Z = torch.empty(1, 2, 0, 32, device="cuda")
    T.ttt_linear_prefill(Z, Z, Z, torch.empty(1, 2, 0, device="cuda"), x["W0"], Z, Wo, 16)
    torch.cuda.synchronize()
    assert torch.equal(Wo, x["W0"])


@pytest.mark.parametrize("kernel", ["fused", "tc", "mma"])
def test_linear_deterministic(kernel):
    x = WL.linear_inputs(2, 3, 256, 64, seed=11, dtype="bf16")
    with linear_kernel(kernel):
        Z1, W1 = run_linear(x, 16)
        Z2, W2 = run_linear(x, 16)
    assert torch.equal(Z1, Z2) and torch.equal(W1, W2)


# -------------------------------------------------------------------- TTT-MLP

MLP_CASES = [(48, 16), (50, 16), (20, 1), (40, 8)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("T_,chunk", MLP_CASES)
def test_mlp_small_shapes(dtype, d, T_, chunk):
    x = WL.mlp_inputs(2, 2, T_, d, 4 * d, seed=200 + d + T_ + chunk, dtype=dtype, w_std=0.1)
    Z, W1, W2 = run_mlp(x, chunk)
    r = f64(x)
    Zr, W1r, W2r = O.mlp_dual(r["Q"], r["K"], r["V"], r["eta"], r["W1"], r["W2"], chunk)
    assert rel_err(Z, Zr) <= TOL[dtype]
    assert rel_err(W1, W1r) <= TOL[dtype]
    assert rel_err(W2, W2r) <= TOL[dtype]


@contextlib.contextmanager
def mlp_kernel(name):
    """Start the TTT-MLP prefill dispatch at kernel `name` ("mma", "tc" or "generic")."""
    old = os.environ.get("TTT_MLP_PREFILL_KERNEL")
    os.environ["TTT_MLP_PREFILL_KERNEL"] = name
    try:
        yield
    finally:
        if old is None:
            del os.environ["TTT_MLP_PREFILL_KERNEL"]
        else:
            os.environ["TTT_MLP_PREFILL_KERNEL"] = old


@pytest.mark.parametrize("kernel", ["mma", "tc"])
@pytest.mark.parametrize("B,H,T_,w_std,seed", [(2, 3, 16, 0.1, 1), (2, 3, 64, 0.02, 2), (2, 3, 400, 0.1, 3),
                                               (2, 3, 1024, 0.05, 4), (4, 50, 48, 0.05, 5)])
def test_mlp_tensor_core_shape(kernel, B, H, T_, w_std, seed):
    # d = 64, hidden = 256, blocks of 16, bf16: the two tensor-core kernels (the last case has
    # more CTAs than SMs)
    x = WL.mlp_inputs(B, H, T_, 64, 256, seed=500 + seed, dtype="bf16", w_std=w_std)
    with mlp_kernel(kernel):
        Z, W1, W2 = run_mlp(x, 16)
    r = f64(x)
    Zr, W1r, W2r = O.mlp_dual(r["Q"], r["K"], r["V"], r["eta"], r["W1"], r["W2"], 16)
    assert rel_err(Z, Zr) <= TOL["bf16"]
    assert rel_err(W1, W1r) <= TOL["bf16"]
    assert rel_err(W2, W2r) <= TOL["bf16"]


@pytest.mark.parametrize("kernel", ["mma", "tc"])
def test_mlp_tensor_core_in_place_split_and_deterministic(kernel, monkeypatch):
    monkeypatch.setenv("TTT_MLP_PREFILL_KERNEL", kernel)
    x = WL.mlp_inputs(1, 4, 128, 64, 256, seed=77, dtype="bf16", w_std=0.1)
    g = cuda(x)
    Z1, A1, B1 = T.mlp_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W1"], g["W2"], 16)
    Z2, A2, B2 = T.mlp_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W1"], g["W2"], 16)
    torch.cuda.synchronize()
    assert torch.equal(Z1, Z2) and torch.equal(A1, A2) and torch.equal(B1, B2)
    # two calls split at a block boundary, chained through the state, updated in place
    W1, W2 = g["W1"].clone(), g["W2"].clone()
    parts = []
    for lo, hi in ((0, 48), (48, 128)):
        sl = lambda t: t[:, :, lo:hi].contiguous()
        Zp = torch.empty_like(sl(g["Q"]))
        T.ttt_mlp_prefill(sl(g["Q"]), sl(g["K"]), sl(g["V"]), sl(g["eta"]), W1, W2, Zp, W1, W2, 16)
        parts.append(Zp)
    torch.cuda.synchronize()
    r = f64(x)
    Zr, W1r, W2r = O.mlp_dual(r["Q"], r["K"], r["V"], r["eta"], r["W1"], r["W2"], 16)
    assert rel_err(torch.cat(parts, 2), Zr) <= TOL["bf16"]
    assert rel_err(W1, W1r) <= TOL["bf16"] and rel_err(W2, W2r) <= TOL["bf16"]
    assert rel_err(Z1, Zr) <= TOL["bf16"]


def test_mlp_prefill_workload_all_heads():
    # B=8 H=12 d=64 hidden=256 T=2048 chunk=16 bf16: all 96 sequences, every element of Z, W1, W2
    w = WL.WORKLOADS["mlp_prefill"]
    x = WL.workload_inputs(w)
    Z, W1, W2 = run_mlp(x, w.chunk)
    r = f64(x)
    Zr, W1r, W2r = O.mlp_dual(r["Q"], r["K"], r["V"], r["eta"], r["W1"], r["W2"], w.chunk)
    check("mlp_prefill B=8 H=12 d=64 h=256 T=2048 b=16", TOL["bf16"], Z=(Z, Zr), W1=(W1, W1r), W2=(W2, W2r))


# ------------------------------------------------------------------- decode

def test_decode_workload_1024_steps():
    # B=256 H=12 d=64: 1024 successive single-token steps on one fp32 state updated in place, as
    # the decode workload states it.  z of every step and the state after the last step against
    # the oracle's online scan (blocks of one token) over the same 1024 tokens, in slices of 32
    # sequences to bound host memory.
    w = WL.WORKLOADS["decode"]
    steps = w.T
    x = WL.decode_inputs(w.B, w.H, w.d, steps, w.seed)
    W = x["W"].cuda()
    q, k, v, e = (x[n].cuda() for n in ("q", "k", "v", "eta"))
    z = torch.empty_like(q)
    for s in range(steps):
        T.ttt_linear_decode_step(q[s], k[s], v[s], e[s], W, z[s])
    torch.cuda.synchronize()
    zc, Wc = z.cpu(), W.cpu()
    del q, k, v, e, z, W
    ez = ew = 0.0
    zmax = wmax = zden = wden = 0.0
    for b0 in range(0, w.B, 32):
        sl = slice(b0, b0 + 32)
        tok = lambda n: WL.to_f64(x[n][:, sl]).transpose(1, 2, 0, 3).copy()  # [steps,b,H,d] -> [b,H,steps,d]
        eta = WL.to_f64(x["eta"][:, sl]).transpose(1, 2, 0).copy()
        Zr, Wr = O.linear_primal(tok("q"), tok("k"), tok("v"), eta, WL.to_f64(x["W"][sl]), 1)
        Zg = zc[:, sl].to(torch.float64).numpy().transpose(1, 2, 0, 3)
        Wg = Wc[sl].to(torch.float64).numpy()
        assert np.all(np.isfinite(Zg)) and np.all(np.isfinite(Wg))
        zmax, zden = max(zmax, float(np.max(np.abs(Zg - Zr)))), max(zden, float(np.max(np.abs(Zr))))
        wmax, wden = max(wmax, float(np.max(np.abs(Wg - Wr)))), max(wden, float(np.max(np.abs(Wr))))
    ez, ew = zmax / zden, wmax / wden
    from tests._parity import MARGINS
    MARGINS.record("decode B=256 H=12 d=64, 1024 steps (z of every step, W after the last)", TOL["bf16"],
                   Z=ez, W=ew)
    assert ez <= TOL["bf16"] and ew <= TOL["bf16"], (ez, ew)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_decode_matches_online_prefill(dtype, d):
    # T decode steps equal a prefill with one-token blocks
    x = WL.linear_inputs(3, 2, 12, d, seed=300 + d, dtype=dtype)
    g = cuda(x)
    W = g["W0"].clone()
    zs = []
    for t in range(12):
        zs.append(T.linear_decode_step(g["Q"][:, :, t].contiguous(), g["K"][:, :, t].contiguous(),
                                       g["V"][:, :, t].contiguous(), g["eta"][:, :, t].contiguous(), W))
    torch.cuda.synchronize()
    r = f64(x)
    Zr, Wr = O.linear_primal(r["Q"], r["K"], r["V"], r["eta"], r["W0"], 1)
    assert rel_err(torch.stack(zs, 2), Zr) <= TOL[dtype]
    assert rel_err(W, Wr) <= TOL[dtype]


# --------------------------------------------------------------- MLP decode

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d,hidden", [(16, 64), (32, 128), (64, 256), (16, 256), (64, 64)])
def test_mlp_decode_steps(dtype, d, hidden):
    steps = 3
    x = WL.mlp_decode_inputs(3, 2, d, hidden, steps, seed=600 + d + hidden, dtype=dtype, w_std=0.1)
    W1, W2 = x["W1"].cuda(), x["W2"].cuda()
    A, Bm = WL.to_f64(x["W1"]), WL.to_f64(x["W2"])
    for s in range(steps):
        q, k, v, e = (x[n][s].cuda() for n in ("q", "k", "v", "eta"))
        z = T.mlp_decode_step(q, k, v, e, W1, W2)
        torch.cuda.synchronize()
        zr, A, Bm = O.mlp_decode(WL.to_f64(x["q"][s]), WL.to_f64(x["k"][s]), WL.to_f64(x["v"][s]),
                                 WL.to_f64(x["eta"][s]), A, Bm)
        assert rel_err(z, zr) <= TOL[dtype]
        assert rel_err(W1, A) <= TOL[dtype]
        assert rel_err(W2, Bm) <= TOL[dtype]


def test_mlp_decode_workload_256_steps():
    # B=64 H=12 d=64 hidden=256: the 256 steps the benchmark's graph runs, W1/W2 in place; z of
    # every step and the state after the last against the oracle's online TTT-MLP scan
    w = WL.WORKLOADS["mlp_decode"]
    steps = w.T
    x = WL.mlp_decode_inputs(w.B, w.H, w.d, w.hidden, steps, w.seed)
    W1, W2 = x["W1"].cuda(), x["W2"].cuda()
    q, k, v, e = (x[n].cuda() for n in ("q", "k", "v", "eta"))
    z = torch.empty_like(q)
    for s in range(steps):
        T.ttt_mlp_decode_step(q[s], k[s], v[s], e[s], W1, W2, z[s])
    torch.cuda.synchronize()
    tok = lambda n: WL.to_f64(x[n]).transpose(1, 2, 0, 3).copy()
    eta = WL.to_f64(x["eta"]).transpose(1, 2, 0).copy()
    Zr, W1r, W2r = O.mlp_primal(tok("q"), tok("k"), tok("v"), eta, WL.to_f64(x["W1"]), WL.to_f64(x["W2"]), 1)
    check("mlp_decode B=64 H=12 d=64 h=256, 256 steps", TOL["bf16"], Z=(z.permute(1, 2, 0, 3), Zr),
          W1=(W1, W1r), W2=(W2, W2r))


def test_mlp_decode_matches_online_prefill():
    # T decode steps equal a TTT-MLP prefill with one-token blocks (both on the GPU)
    x = WL.mlp_inputs(2, 3, 10, 32, 128, seed=610, dtype="f32", w_std=0.1)
    g = cuda(x)
    Zp, W1p, W2p = T.mlp_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W1"], g["W2"], 1)
    W1, W2 = g["W1"].clone(), g["W2"].clone()
    zs = [T.mlp_decode_step(g["Q"][:, :, t].contiguous(), g["K"][:, :, t].contiguous(), g["V"][:, :, t].contiguous(),
                            g["eta"][:, :, t].contiguous(), W1, W2) for t in range(10)]
    torch.cuda.synchronize()
    r = f64(x)
    Zr, W1r, W2r = O.mlp_primal(r["Q"], r["K"], r["V"], r["eta"], r["W1"], r["W2"], 1)
    assert rel_err(torch.stack(zs, 2), Zr) <= TOL["f32"] and rel_err(Zp, Zr) <= TOL["f32"]
    assert rel_err(W1, W1r) <= TOL["f32"] and rel_err(W2, W2r) <= TOL["f32"]


# ------------------------------------------------- prefill -> decode hand-off

@pytest.mark.parametrize("kind", ["linear", "mlp"])
def test_prefill_then_decode_hand_off(kind):
    # a prompt of P tokens in blocks of 16 (last block ragged), then D single-token decode steps
    # from the prefill's final state: the oracle runs the same schedule (block scan, then b = 1)
    P, Dn, d = 40, 5, 64
    if kind == "linear":
        x = WL.linear_inputs(2, 3, P + Dn, d, seed=700, dtype="bf16")
    else:
        x = WL.mlp_inputs(2, 3, P + Dn, d, 256, seed=701, dtype="bf16", w_std=0.1)
    g = cuda(x)
    sl = lambda t, a, b: t[:, :, a:b].contiguous()
    r = f64(x)
    rs = lambda t, a, b: t[:, :, a:b]
    if kind == "linear":
        Zp, W = T.linear_prefill(sl(g["Q"], 0, P), sl(g["K"], 0, P), sl(g["V"], 0, P), sl(g["eta"], 0, P), g["W0"], 16)
        zs = [T.linear_decode_step(g["Q"][:, :, t].contiguous(), g["K"][:, :, t].contiguous(),
                                   g["V"][:, :, t].contiguous(), g["eta"][:, :, t].contiguous(), W)
              for t in range(P, P + Dn)]
        torch.cuda.synchronize()
        Zr1, Wr1 = O.linear_primal(rs(r["Q"], 0, P), rs(r["K"], 0, P), rs(r["V"], 0, P), rs(r["eta"], 0, P), r["W0"], 16)
        Zr2, Wr2 = O.linear_primal(rs(r["Q"], P, P + Dn), rs(r["K"], P, P + Dn), rs(r["V"], P, P + Dn),
                                   rs(r["eta"], P, P + Dn), Wr1, 1)
        assert rel_err(W, Wr2) <= TOL["bf16"]
    else:
        Zp, W1, W2 = T.mlp_prefill(sl(g["Q"], 0, P), sl(g["K"], 0, P), sl(g["V"], 0, P), sl(g["eta"], 0, P),
                                   g["W1"], g["W2"], 16)
        zs = [T.mlp_decode_step(g["Q"][:, :, t].contiguous(), g["K"][:, :, t].contiguous(),
                                g["V"][:, :, t].contiguous(), g["eta"][:, :, t].contiguous(), W1, W2)
              for t in range(P, P + Dn)]
        torch.cuda.synchronize()
        Zr1, A1, B1 = O.mlp_primal(rs(r["Q"], 0, P), rs(r["K"], 0, P), rs(r["V"], 0, P), rs(r["eta"], 0, P),
                                   r["W1"], r["W2"], 16)
        Zr2, A2, B2 = O.mlp_primal(rs(r["Q"], P, P + Dn), rs(r["K"], P, P + Dn), rs(r["V"], P, P + Dn),
                                   rs(r["eta"], P, P + Dn), A1, B1, 1)
        assert rel_err(W1, A2) <= TOL["bf16"] and rel_err(W2, B2) <= TOL["bf16"]
    assert rel_err(Zp, Zr1) <= TOL["bf16"]
    assert rel_err(torch.stack(zs, 2), Zr2) <= TOL["bf16"]


# bf16 with 16 | T but chunk not dividing T: the tensor-core kernels take the shorter last block as fewer
# 16-token sub-blocks
@pytest.mark.parametrize("d,kernel", [(64, "fused"), (64, "mma"), (128, "mma")])
@pytest.mark.parametrize("B,H,T_,chunk", [(2, 3, 208, 64), (1, 2, 1040, 512), (2, 2, 96, 80), (3, 16, 272, 32)])
def test_linear_tensor_core_kernels_ragged_last_block(d, kernel, B, H, T_, chunk):
    x = WL.linear_inputs(B, H, T_, d, seed=900 + T_ + chunk + d, dtype="bf16")
    with linear_kernel(kernel):
        Z, W = run_linear(x, chunk)
    r = f64(x)
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], chunk)
    assert rel_err(Z, Zr) <= TOL["bf16"]
    assert rel_err(W, Wr) <= TOL["bf16"]


# bf16, T not a multiple of 16: the tensor-core kernels run a partial last sub-block (its eta from
# global memory, read only where the tokens exist; with 4 not dividing T every sub-block's eta comes
# from there).  T = 260 / 261 leave the fused kernel's last stage of 256 tokens holding only the
# partial sub-block; T = 67 / 68 do the same for the split kernel's stages of 64 tokens at d = 128.
@pytest.mark.parametrize("d,kernel", [(64, "fused"), (64, "mma"), (128, "mma")])
@pytest.mark.parametrize("T_", [1, 7, 17, 67, 68, 203, 212, 260, 261, 2047])
@pytest.mark.parametrize("chunk", [16, 64])
def test_tensor_core_partial_last_sub_block(d, kernel, T_, chunk):
    x = WL.linear_inputs(2, 3, T_, d, seed=950 + T_ + chunk + d, dtype="bf16")
    with linear_kernel(kernel):
        Z, W = run_linear(x, chunk)
    r = f64(x)
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], chunk)
    assert rel_err(Z, Zr) <= TOL["bf16"]
    assert rel_err(W, Wr) <= TOL["bf16"]


@pytest.mark.parametrize("d,kernel", [(64, "fused"), (128, "mma")])
def test_partial_sub_block_reads_no_rows_of_the_next_head(d, kernel):
    # head 1 holds values whose products overflow; head 0 (T = 23: a partial second sub-block) must
    # not see them, since the tokens past its end read as zeros rather than as head 1's rows
    x = WL.linear_inputs(1, 2, 23, d, seed=977, dtype="bf16")
    for k in ("Q", "K", "V"):
        x[k][:, 1] = 3.0e38
    with linear_kernel(kernel):
        Z, W = run_linear(x, 16)
    r = f64({k: v[:, :1] for k, v in x.items()})
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], 16)
    assert rel_err(Z[:, :1], Zr) <= TOL["bf16"]
    assert rel_err(W[:, :1], Wr) <= TOL["bf16"]


# TTT-MLP, bf16, d = 64, hidden = 256, blocks of 16, T not a multiple of 16: the warp-MMA kernel runs
# a partial last block (its eta stored by the producer thread, zero past T; with 4 not dividing T
# every block's eta is stored that way)
@pytest.mark.parametrize("T_", [1, 7, 17, 50, 203, 1001])
def test_mlp_mma_partial_last_block(T_):
    x = WL.mlp_inputs(2, 3, T_, 64, 256, seed=520 + T_, dtype="bf16", w_std=0.05)
    with mlp_kernel("mma"):
        Z, W1, W2 = run_mlp(x, 16)
    r = f64(x)
    Zr, W1r, W2r = O.mlp_dual(r["Q"], r["K"], r["V"], r["eta"], r["W1"], r["W2"], 16)
    assert rel_err(Z, Zr) <= TOL["bf16"]
    assert rel_err(W1, W1r) <= TOL["bf16"]
    assert rel_err(W2, W2r) <= TOL["bf16"]


def test_mlp_mma_partial_block_reads_no_rows_of_the_next_head():
    # head 1 holds values whose products overflow; head 0 (T = 21) must not see them
    x = WL.mlp_inputs(1, 2, 21, 64, 256, seed=531, dtype="bf16", w_std=0.05)
    for k in ("Q", "K", "V"):
        x[k][:, 1] = 3.0e38
    with mlp_kernel("mma"):
        Z, W1, W2 = run_mlp(x, 16)
    r = f64({k: v[:, :1] for k, v in x.items()})
    Zr, W1r, W2r = O.mlp_dual(r["Q"], r["K"], r["V"], r["eta"], r["W1"], r["W2"], 16)
    assert rel_err(Z[:, :1], Zr) <= TOL["bf16"]
    assert rel_err(W1[:, :1], W1r) <= TOL["bf16"] and rel_err(W2[:, :1], W2r) <= TOL["bf16"]
