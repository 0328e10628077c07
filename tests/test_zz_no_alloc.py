"""The split TTT-Linear prefill with the library's built-in scratch (ttt_linear_prefill_noalloc),
for callers that cannot allocate device memory when they run the scan: through the C ABI, its output
must match the same split computed with caller-owned scratch (ttt_linear_prefill_ws), on two calls in
a row with different inputs (the scratch keeps the previous call's contents, which must not leak into
the next result).  Collected last on purpose (file name), and independent of every other test file.
"""
import pytest
import torch

from test_sequence_layers_07_b300 import ttt as T
from test_sequence_layers_07_b300 import workloads as WL
from tests._parity import TOL, cuda

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))


def test_noalloc_matches_caller_scratch_on_two_calls(monkeypatch):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    T.load_library()
    monkeypatch.delenv("TTT_LINEAR_SEGMENTS", raising=False)
    w = WL.WORKLOADS["linear_few_heads"]  # 4 heads, 16384 tokens: split, 12.6 MB of scratch
    need = T.ttt_linear_prefill_workspace_size(w.B, w.H, w.T, w.d, w.chunk, torch.bfloat16)
    assert 0 < need <= SCRATCH_BYTES
    # two calls in a row on different inputs; every tensor exists before the first call
    runs = []
    for seed in (w.seed, w.seed + 1):
        g = cuda(WL.linear_inputs(w.B, w.H, w.T, w.d, seed=seed, dtype=w.dtype))
        ref = T.linear_prefill_ws(g["Q"], g["K"], g["V"], g["eta"], g["W0"], w.chunk)  # caller-owned scratch
        runs.append((g, torch.empty_like(g["Q"]), torch.empty_like(g["W0"]), ref))
    torch.cuda.synchronize()
    free = []
    for g, Z, W, _ in runs:
        T.ttt_linear_prefill_noalloc(g["Q"], g["K"], g["V"], g["eta"], g["W0"], Z, W, w.chunk)
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
    for g, Z, W, (Zw, Ww) in runs:
        assert torch.isfinite(Z.float()).all() and torch.isfinite(W).all()
        assert _rel(Z, Zw) <= TOL["bf16"] and _rel(W, Ww) <= TOL["bf16"]
    # the second call allocated nothing on the device (the first may load the library's module)
    assert free[1] >= free[0] - (2 << 20)
    assert T.ttt_get_device_status() == T.TTT_OK


def test_noalloc_rejects_a_split_larger_than_its_scratch(monkeypatch):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    T.load_library()
    # 200 segments of 4 heads at d = 64: 4 * (3 * 200 - 2) * 16 KB = 39 MB of maps and start states
    monkeypatch.setenv("TTT_LINEAR_SEGMENTS", "200")
    x = WL.linear_inputs(1, 4, 3200, 64, seed=5, dtype="bf16")
    assert T.ttt_linear_prefill_workspace_size(1, 4, 3200, 64, 16, torch.bfloat16) > SCRATCH_BYTES
    g = cuda(x)
    Z, W = torch.empty_like(g["Q"]), torch.empty_like(g["W0"])
    with pytest.raises(T.TTTError) as err:
        T.ttt_linear_prefill_noalloc(g["Q"], g["K"], g["V"], g["eta"], g["W0"], Z, W, 16)
    assert err.value.status == T.TTT_ERR_UNSUPPORTED and "scratch" in str(err.value)
