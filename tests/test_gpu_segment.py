"""GPU parity of the TTT-Linear prefill split along the sequence (ttt_linear_prefill_ws) against
the fp64 oracle, through the C ABI: each stage's workspace contents (segment maps, start states) and
the results (Z, final state).

The oracle pins what each stage means without sharing anything with the kernels:
  * Delta_s + I is the state a segment reaches from W = I with targets V = 0 (the segment's linear
    part), and B_s the state it reaches from W = 0 with the real V;
  * the start state of segment s is the final state of the one-pass scan over the tokens before it.
Error metric max|delta| / ||ref||_inf per output, bar 2e-2 (bf16 inputs).
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


def plan(T_, chunk, S_req):
    """Segment length (tokens) and count for an explicit request of S_req segments."""
    nblk = T_ // chunk
    L = -(-nblk // S_req)
    return L * chunk, -(-nblk // L)


def run_ws(x, chunk, S_req, monkeypatch, in_place=False):
    monkeypatch.setenv("TTT_LINEAR_SEGMENTS", str(S_req))
    g = cuda(x)
    B, H, T_, d = g["Q"].shape
    n = T.ttt_linear_prefill_workspace_size(B, H, T_, d, chunk, g["Q"].dtype)
    ws = torch.full((max(n, 4) // 4,), float("nan"), device="cuda") if n else None
    Z = torch.empty_like(g["Q"])
    W = g["W0"].clone() if in_place else torch.empty_like(g["W0"])
    W0 = W if in_place else g["W0"]
    T.ttt_linear_prefill_ws(g["Q"], g["K"], g["V"], g["eta"], W0, Z, W, chunk, ws)
    torch.cuda.synchronize()
    return Z, W, ws


def split_ws(ws, B, H, d, S):
    P = B * H
    nm = P * (S - 1) * 2 * d * d
    maps = ws[:nm].view(B, H, S - 1, 2, d, d)
    starts = ws[nm:nm + P * S * d * d].view(B, H, S, d, d)
    return maps, starts


SEG_CASES = [  # B, H, T, chunk, segments asked for
    (2, 3, 512, 16, 2),
    (2, 3, 512, 16, 3),      # 32 blocks in segments of 11, 11, 10
    (1, 4, 1024, 64, 5),     # blocks of 64 (four sub-blocks)
    (2, 2, 640, 32, 4),      # 20 blocks of 32 in 4 segments of 5
    (1, 2, 2048, 256, 8),    # one block per segment
    (1, 3, 160, 16, 10),     # one block per segment, 10 segments
    (3, 50, 256, 16, 2),     # 300 (head, segment) pairs: more CTAs than SMs
]


@pytest.mark.parametrize("B,H,T_,chunk,S_req", SEG_CASES)
def test_segment_stages_and_results(B, H, T_, chunk, S_req, monkeypatch):
    d = 64
    x = WL.linear_inputs(B, H, T_, d, seed=2000 + T_ + chunk + S_req, dtype="bf16", w_std=0.05)
    Z, W, ws = run_ws(x, chunk, S_req, monkeypatch)
    seg_len, S = plan(T_, chunk, S_req)
    r = f64(x)
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], chunk)
    assert rel_err(Z, Zr) <= TOL["bf16"] and rel_err(W, Wr) <= TOL["bf16"]
    assert ws is not None and ws.numel() * 4 == B * H * (3 * S - 2) * d * d * 4
    maps, starts = split_ws(ws, B, H, d, S)
    eye = np.broadcast_to(np.eye(d), (B, H, d, d))
    for s in range(S):
        t0, t1 = s * seg_len, min(T_, (s + 1) * seg_len)
        # start state: the one-pass scan over the tokens before the segment
        if s == 0:
            assert torch.equal(starts[:, :, 0], x["W0"].cuda())
        else:
            pre = {k: (v[:, :, :t0] if k != "W0" else v) for k, v in r.items()}
            _, Ws = O.linear_dual(pre["Q"], pre["K"], pre["V"], pre["eta"], pre["W0"], chunk)
            assert rel_err(starts[:, :, s], Ws) <= TOL["bf16"], s
        if s == S - 1:
            continue
        seg = {k: (v[:, :, t0:t1] if k != "W0" else v) for k, v in r.items()}
        _, A = O.linear_dual(seg["Q"], seg["K"], np.zeros_like(seg["V"]), seg["eta"], eye.copy(), chunk)
        _, Bs = O.linear_dual(seg["Q"], seg["K"], seg["V"], seg["eta"], np.zeros_like(seg["W0"]), chunk)
        assert rel_err(maps[:, :, s, 0], A - eye) <= TOL["bf16"], ("Delta", s)
        assert rel_err(maps[:, :, s, 1], Bs) <= TOL["bf16"], ("B", s)


def test_segment_in_place_state_and_deterministic(monkeypatch):
    x = WL.linear_inputs(2, 6, 768, 64, seed=2100, dtype="bf16")
    Z1, W1, _ = run_ws(x, 16, 3, monkeypatch)
    Z2, W2, _ = run_ws(x, 16, 3, monkeypatch, in_place=True)
    assert torch.equal(Z1, Z2) and torch.equal(W1, W2)
    Z3, W3, _ = run_ws(x, 16, 3, monkeypatch)
    assert torch.equal(Z1, Z3) and torch.equal(W1, W3)
    r = f64(x)
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], 16)
    assert rel_err(Z1, Zr) <= TOL["bf16"] and rel_err(W1, Wr) <= TOL["bf16"]


def test_segment_shapes_outside_the_split_run_the_one_pass_scan(monkeypatch):
    # fp32 and d = 128: workspace size 0, the call is the one-pass prefill (no workspace needed)
    monkeypatch.delenv("TTT_LINEAR_SEGMENTS", raising=False)
    for d, dtype in ((64, "f32"), (128, "bf16"), (32, "bf16")):
        x = WL.linear_inputs(1, 2, 96, d, seed=2200 + d, dtype=dtype)
        g = cuda(x)
        assert T.ttt_linear_prefill_workspace_size(1, 2, 96, d, 16, g["Q"].dtype) == 0
        Z, W = T.linear_prefill_ws(g["Q"], g["K"], g["V"], g["eta"], g["W0"], 16)
        torch.cuda.synchronize()
        r = f64(x)
        Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], 16)
        assert rel_err(Z, Zr) <= TOL[dtype] and rel_err(W, Wr) <= TOL[dtype]


def test_linear_prefill_ws_few_heads_workload_all_heads(monkeypatch):
    # B=1 H=4 d=64 T=16384 chunk=16 bf16 (few heads, long prompt), in the segment plan the library
    # chooses from the SM count and the benchmark times: every element of Z and of the final state
    monkeypatch.delenv("TTT_LINEAR_SEGMENTS", raising=False)
    w = WL.WORKLOADS["linear_few_heads"]
    x = WL.workload_inputs(w)
    g = cuda(x)
    assert T.ttt_linear_prefill_workspace_size(w.B, w.H, w.T, w.d, w.chunk, g["Q"].dtype) > 0
    Z, W = T.linear_prefill_ws(g["Q"], g["K"], g["V"], g["eta"], g["W0"], w.chunk)
    torch.cuda.synchronize()
    r = f64(x)
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], w.chunk)
    check("linear_prefill split along the sequence, B=1 H=4 d=64 T=16384 b=16", TOL["bf16"], Z=(Z, Zr),
          W=(W, Wr))


def test_linear_prefill_ws_headline_runs_one_pass(monkeypatch):
    # the headline shape needs no workspace (one pass); the call through the split entry point matches
    monkeypatch.delenv("TTT_LINEAR_SEGMENTS", raising=False)
    w = WL.WORKLOADS["linear_prefill"]
    x = WL.linear_inputs(w.B, w.H, 256, w.d, seed=w.seed, dtype=w.dtype)
    g = cuda(x)
    assert T.ttt_linear_prefill_workspace_size(w.B, w.H, w.T, w.d, w.chunk, g["Q"].dtype) == 0
    Z, W = T.linear_prefill_ws(g["Q"], g["K"], g["V"], g["eta"], g["W0"], w.chunk)
    Z1, W1 = T.linear_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W0"], w.chunk)
    torch.cuda.synchronize()
    assert torch.equal(Z, Z1) and torch.equal(W, W1)
