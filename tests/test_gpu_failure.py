"""Device-side failure detection, without a GPU fault.

A kernel waits, with the library's bounded wait, on a barrier that nothing
completes.  After its limit it records TTT_ERR_TIMEOUT in the device status
word and returns; the host reads the status, which is then cleared, and the
context keeps working (a prefill afterwards matches the oracle).
"""
import pytest
import torch

from oracle import oracle as O
from test_sequence_layers_07_b300 import ttt as T
from test_sequence_layers_07_b300 import workloads as WL
from tests._parity import TOL, cuda, f64, rel_err

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_context_survives():
    assert torch.cuda.is_available()
    T.load_library()
    assert T.ttt_get_device_status() == T.TTT_OK  # nothing pending
    T.ttt_selftest_wait_timeout(2_000_000)  # 2 ms
    assert T.ttt_get_device_status() == T.TTT_ERR_TIMEOUT
    assert T.ttt_get_device_status() == T.TTT_OK  # read-and-clear
    # the context is intact: a normal call still runs and is correct
    x = WL.linear_inputs(1, 2, 64, 64, seed=5, dtype="bf16")
    g = cuda(x)
    Z, W = T.linear_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W0"], 16)
    torch.cuda.synchronize()
    r = f64(x)
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], 16)
    assert rel_err(Z, Zr) <= TOL["bf16"] and rel_err(W, Wr) <= TOL["bf16"]
    assert T.ttt_get_device_status() == T.TTT_OK


def test_prefill_wait_expiry_is_reported_and_context_survives(monkeypatch):
    # A real TTT-Linear prefill (the d = 64 fused kernel) with its barrier waits bounded at 1 ns:
    # the producer's wait for a stage the column-group warps still read must expire (a stage takes
    # microseconds), so the kernel records TTT_ERR_TIMEOUT, every warp leaves its loop, the copies
    # in flight are drained, and the context stays usable.
    assert torch.cuda.is_available()
    T.load_library()
    assert T.ttt_get_device_status() == T.TTT_OK
    x = WL.linear_inputs(2, 12, 2048, 64, seed=6, dtype="bf16")
    g = cuda(x)
    monkeypatch.setenv("TTT_WAIT_LIMIT_NS", "1")
    T.linear_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W0"], 16)
    torch.cuda.synchronize()
    monkeypatch.delenv("TTT_WAIT_LIMIT_NS")
    assert T.ttt_get_device_status() == T.TTT_ERR_TIMEOUT
    assert T.ttt_get_device_status() == T.TTT_OK
    Z, W = T.linear_prefill(g["Q"], g["K"], g["V"], g["eta"], g["W0"], 16)
    torch.cuda.synchronize()
    assert T.ttt_get_device_status() == T.TTT_OK
    r = f64(x)
    Zr, Wr = O.linear_dual(r["Q"], r["K"], r["V"], r["eta"], r["W0"], 16)
    assert rel_err(Z, Zr) <= TOL["bf16"] and rel_err(W, Wr) <= TOL["bf16"]
