"""Host-side checks of the C ABI (no GPU needed).

* libttt.so loads and exports every function include/ttt.h declares;
* argument validation returns the documented status before any CUDA call
  (null or misaligned pointers, negative sizes, bad chunk, unsupported d);
* empty problems (B*H == 0) return TTT_OK without touching the device.
"""
import ctypes
import os
import re
import subprocess

import pytest

from test_sequence_layers_07_b300 import build as B
from test_sequence_layers_07_b300 import ttt as T

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ttt.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(T.LIB_PATH):
        B.build()
    return T.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ttt_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_documented_entry_points():
    names = declared_functions()
    for n in ("ttt_linear_prefill", "ttt_mlp_prefill", "ttt_linear_decode_step", "ttt_get_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", T.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (ttt_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)
    assert set(T.EXPORTED) == set(declared_functions())


def test_header_compiles_as_c():
    r = subprocess.run(["gcc", "-x", "c", "-std=c99", "-fsyntax-only", "-Wall", "-Werror", HEADER],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_status_strings(lib):
    assert lib.ttt_status_string(0) == b"ok"
    assert lib.ttt_status_string(1) == b"invalid argument"
    assert lib.ttt_status_string(4) == b"device-side wait timed out"
    assert lib.ttt_version() >= 100


# fake 16-byte-aligned addresses: validation must reject the call before using them
A = 0x10000
MIS = 0x10008
NULL = None


def lp(lib, Q=A, K=A, V=A, eta=A, W0=A, Z=A, Wo=A, B_=1, H=1, T_=16, d=64, chunk=16, dt=1):
    return lib.ttt_linear_prefill(Q, K, V, eta, W0, Z, Wo, B_, H, T_, d, chunk, dt, None)


def test_linear_prefill_validation(lib):
    assert lp(lib, Q=NULL) == T.TTT_ERR_INVALID_ARG
    assert b"Q" in lib.ttt_last_error()
    assert lp(lib, W0=NULL) == T.TTT_ERR_INVALID_ARG
    assert lp(lib, Z=MIS) == T.TTT_ERR_INVALID_ARG
    assert b"aligned" in lib.ttt_last_error()
    assert lp(lib, B_=-1) == T.TTT_ERR_INVALID_ARG
    assert lp(lib, T_=-3) == T.TTT_ERR_INVALID_ARG
    assert lp(lib, chunk=0) == T.TTT_ERR_INVALID_ARG
    assert lp(lib, chunk=513) == T.TTT_ERR_INVALID_ARG
    assert lp(lib, dt=7) == T.TTT_ERR_INVALID_ARG
    assert lp(lib, d=0) == T.TTT_ERR_INVALID_ARG
    assert lp(lib, d=48) == T.TTT_ERR_UNSUPPORTED
    assert lp(lib, d=256) == T.TTT_ERR_UNSUPPORTED
    # empty batch: nothing to do, no device access even with null pointers
    assert lp(lib, Q=NULL, K=NULL, V=NULL, eta=NULL, W0=NULL, Z=NULL, Wo=NULL, B_=0) == T.TTT_OK
    assert lp(lib, Q=NULL, K=NULL, V=NULL, eta=NULL, W0=NULL, Z=NULL, Wo=NULL, H=0) == T.TTT_OK


def test_linear_prefill_hist_validation(lib):
    def hp(Q=A, K=A, V=A, eta=A, W0=A, Z=A, Wo=A, Wh=A, B_=1, H=1, T_=16, d=64, chunk=16, dt=1):
        return lib.ttt_linear_prefill_hist(Q, K, V, eta, W0, Z, Wo, Wh, B_, H, T_, d, chunk, dt, None)

    assert hp(Wh=NULL) == T.TTT_ERR_INVALID_ARG
    assert b"W_hist" in lib.ttt_last_error()
    assert hp(Wh=MIS) == T.TTT_ERR_INVALID_ARG
    assert hp(K=NULL) == T.TTT_ERR_INVALID_ARG
    assert hp(chunk=0) == T.TTT_ERR_INVALID_ARG
    assert hp(d=48) == T.TTT_ERR_UNSUPPORTED
    assert hp(Q=NULL, K=NULL, V=NULL, eta=NULL, W0=NULL, Z=NULL, Wo=NULL, Wh=NULL, B_=0) == T.TTT_OK


def test_linear_backward_validation(lib):
    def bp(Q=A, K=A, V=A, eta=A, Wh=A, dZ=A, dWT=A, dQ=A, dK=A, dV=A, de=A, dW0=A, B_=1, H=1, T_=16, d=64,
           chunk=16, dt=1):
        return lib.ttt_linear_prefill_backward(Q, K, V, eta, Wh, dZ, dWT, dQ, dK, dV, de, dW0, B_, H, T_, d,
                                               chunk, dt, None)

    assert bp(dZ=NULL) == T.TTT_ERR_INVALID_ARG
    assert b"dZ" in lib.ttt_last_error()
    assert bp(Wh=NULL) == T.TTT_ERR_INVALID_ARG
    assert bp(de=MIS) == T.TTT_ERR_INVALID_ARG
    assert bp(dWT=MIS) == T.TTT_ERR_INVALID_ARG
    assert bp(dW0=NULL) == T.TTT_ERR_INVALID_ARG
    assert bp(B_=-1) == T.TTT_ERR_INVALID_ARG
    assert bp(chunk=513) == T.TTT_ERR_INVALID_ARG
    assert bp(dt=3) == T.TTT_ERR_INVALID_ARG
    assert bp(d=96) == T.TTT_ERR_UNSUPPORTED
    # block tiles beyond shared memory: d = 64 takes chunk <= 64, d = 128 chunk <= 16
    assert bp(chunk=128) == T.TTT_ERR_UNSUPPORTED
    assert bp(d=128, chunk=32) == T.TTT_ERR_UNSUPPORTED
    assert b"shared memory" in lib.ttt_last_error()
    assert bp(Q=NULL, K=NULL, V=NULL, eta=NULL, Wh=NULL, dZ=NULL, dWT=NULL, dQ=NULL, dK=NULL, dV=NULL, de=NULL,
              dW0=NULL, H=0) == T.TTT_OK


def test_mlp_prefill_validation(lib):
    def mp(**kw):
        a = dict(Q=A, K=A, V=A, eta=A, W1=A, W2=A, Z=A, W1o=A, W2o=A, B_=1, H=1, T_=16, d=64, hd=256, chunk=16,
                 dt=1)
        a.update(kw)
        return lib.ttt_mlp_prefill(a["Q"], a["K"], a["V"], a["eta"], a["W1"], a["W2"], a["Z"], a["W1o"], a["W2o"],
                                   a["B_"], a["H"], a["T_"], a["d"], a["hd"], a["chunk"], a["dt"], None)
    assert mp(W2=NULL) == T.TTT_ERR_INVALID_ARG
    assert mp(W1o=MIS) == T.TTT_ERR_INVALID_ARG
    assert mp(chunk=0) == T.TTT_ERR_INVALID_ARG
    assert mp(d=128, hd=512) == T.TTT_ERR_UNSUPPORTED
    assert mp(hd=250) == T.TTT_ERR_UNSUPPORTED
    assert mp(chunk=32) == T.TTT_ERR_UNSUPPORTED  # chunk*hidden > 4096
    assert mp(hd=0) == T.TTT_ERR_INVALID_ARG
    assert mp(B_=0, Q=NULL, W1=NULL) == T.TTT_OK


def test_decode_validation(lib):
    def dp(**kw):
        a = dict(q=A, k=A, v=A, eta=A, W=A, z=A, B_=2, H=3, d=64, dt=1)
        a.update(kw)
        return lib.ttt_linear_decode_step(a["q"], a["k"], a["v"], a["eta"], a["W"], a["z"], a["B_"], a["H"], a["d"],
                                          a["dt"], None)
    assert dp(W=NULL) == T.TTT_ERR_INVALID_ARG
    assert dp(eta=MIS) == T.TTT_ERR_INVALID_ARG
    assert dp(d=40) == T.TTT_ERR_UNSUPPORTED
    assert dp(H=-1) == T.TTT_ERR_INVALID_ARG
    assert dp(B_=0, W=NULL) == T.TTT_OK


def test_mlp_decode_validation(lib):
    def md(**kw):
        a = dict(q=A, k=A, v=A, eta=A, W1=A, W2=A, z=A, B_=2, H=3, d=64, hd=256, dt=1)
        a.update(kw)
        return lib.ttt_mlp_decode_step(a["q"], a["k"], a["v"], a["eta"], a["W1"], a["W2"], a["z"], a["B_"], a["H"],
                                       a["d"], a["hd"], a["dt"], None)
    assert md(W2=NULL) == T.TTT_ERR_INVALID_ARG
    assert b"W2" in lib.ttt_last_error()
    assert md(z=MIS) == T.TTT_ERR_INVALID_ARG
    assert md(d=128) == T.TTT_ERR_UNSUPPORTED
    assert md(hd=192) == T.TTT_ERR_UNSUPPORTED
    assert md(hd=0) == T.TTT_ERR_INVALID_ARG
    assert md(dt=3) == T.TTT_ERR_INVALID_ARG
    assert md(B_=-2) == T.TTT_ERR_INVALID_ARG
    assert md(H=0, W1=NULL, W2=NULL) == T.TTT_OK


def test_selftest_limit_validation(lib):
    assert lib.ttt_selftest_wait_timeout(0, None) == T.TTT_ERR_INVALID_ARG
    assert lib.ttt_selftest_wait_timeout(3 * 10**9, None) == T.TTT_ERR_INVALID_ARG


def test_binding_rejects_cpu_tensors(lib):
    import torch
    x = torch.zeros(1, 1, 16, 16)
    with pytest.raises((TypeError, ValueError)):
        T.ttt_linear_prefill(x, x, x, torch.zeros(1, 1, 16), torch.zeros(1, 1, 16, 16), x, torch.zeros(1, 1, 16, 16), 16)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(FileNotFoundError):
        # a fresh loader pointed at a path with no library must raise, not fall back
        import importlib
        mod = importlib.import_module("test_sequence_layers_07_b300.ttt")
        saved = mod._lib
        try:
            mod._lib = None
            mod.load_library(str(tmp_path / "libttt.so"))
        finally:
            mod._lib = saved


def test_linear_prefill_ws_sizes_and_validation(lib, monkeypatch):
    monkeypatch.delenv("TTT_LINEAR_SEGMENTS", raising=False)
    ws = lib.ttt_linear_prefill_workspace_size
    unit = 64 * 64 * 4
    # the headline shape (96 heads) fills most SMs in one pass: not split
    assert ws(8, 12, 2048, 64, 16, 1) == 0
    n = ws(1, 4, 16384, 64, 16, 1)  # four heads, long prompt: split into segments of >= 256 tokens
    assert n > 0 and n % (4 * unit) == 0
    S = (n // (4 * unit) + 2) // 3
    assert n == 4 * (3 * S - 2) * unit and 2 <= S <= 16384 // 256
    # shapes outside the split, or too short to split: 0 (the call is the one-pass scan)
    assert ws(8, 12, 2048, 64, 16, 0) == 0        # fp32
    assert ws(8, 12, 2048, 128, 16, 1) == 0       # d = 128
    assert ws(8, 12, 2048, 64, 8, 1) == 0         # chunk not a multiple of 16
    assert ws(8, 12, 2000, 64, 48, 1) == 0        # chunk does not divide T
    assert ws(1, 1, 255, 64, 1, 1) == 0
    assert ws(1, 1, 128, 64, 16, 1) == 0          # under 256 tokens: one segment
    assert ws(0, 12, 2048, 64, 16, 1) == 0 and ws(8, 12, 0, 64, 16, 1) == 0
    # an explicit segment count: 10 blocks of 16 in 3 segments of 4, 4, 2 blocks
    monkeypatch.setenv("TTT_LINEAR_SEGMENTS", "3")
    assert ws(2, 3, 160, 64, 16, 1) == 6 * (3 * 3 - 2) * unit
    monkeypatch.setenv("TTT_LINEAR_SEGMENTS", "4")  # 10 blocks: segments of 3 -> 4 segments
    assert ws(2, 3, 160, 64, 16, 1) == 6 * (3 * 4 - 2) * unit
    monkeypatch.setenv("TTT_LINEAR_SEGMENTS", "6")  # segments of 2 blocks -> 5 segments
    assert ws(2, 3, 160, 64, 16, 1) == 6 * (3 * 5 - 2) * unit
    monkeypatch.setenv("TTT_LINEAR_SEGMENTS", "1")
    assert ws(8, 12, 2048, 64, 16, 1) == 0
    monkeypatch.delenv("TTT_LINEAR_SEGMENTS")

    def call(workspace=A, nbytes=n, Q=A, **kw):
        return lib.ttt_linear_prefill_ws(Q, A, A, A, A, A, A, 1, 4, 16384, 64, 16, 1, workspace, nbytes, None)

    assert call(nbytes=n - 16) == T.TTT_ERR_INVALID_ARG
    assert b"workspace" in lib.ttt_last_error()
    assert call(workspace=NULL) == T.TTT_ERR_INVALID_ARG
    assert call(workspace=MIS) == T.TTT_ERR_INVALID_ARG
    assert call(Q=NULL) == T.TTT_ERR_INVALID_ARG
    assert lib.ttt_linear_prefill_ws(A, A, A, A, A, A, A, 1, 4, 16384, 48, 16, 1, A, n, None) == T.TTT_ERR_UNSUPPORTED
    # nothing to do: no device access even with null pointers and no workspace
    assert lib.ttt_linear_prefill_ws(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 12, 2048, 64, 16, 1, NULL, 0,
                                     None) == T.TTT_OK


def test_linear_momentum_validation(lib):
    import ctypes

    def mp(Q=A, M0=A, Mo=A, B_=1, H=1, T_=16, d=64, chunk=16, beta=0.9, dt=1):
        return lib.ttt_linear_momentum_prefill(Q, A, A, A, A, M0, A, A, Mo, B_, H, T_, d, chunk, ctypes.c_float(beta),
                                               dt, None)

    assert mp(beta=-0.1) == T.TTT_ERR_INVALID_ARG
    assert b"beta" in lib.ttt_last_error()
    assert mp(beta=1.5) == T.TTT_ERR_INVALID_ARG
    assert mp(beta=float("nan")) == T.TTT_ERR_INVALID_ARG
    assert mp(Mo=NULL) == T.TTT_ERR_INVALID_ARG
    assert mp(M0=MIS) == T.TTT_ERR_INVALID_ARG
    assert mp(Q=NULL) == T.TTT_ERR_INVALID_ARG
    assert mp(chunk=0) == T.TTT_ERR_INVALID_ARG
    assert mp(d=48) == T.TTT_ERR_UNSUPPORTED
    assert mp(Q=NULL, M0=NULL, Mo=NULL, B_=0) == T.TTT_OK


def test_mlp_hist_and_backward_validation(lib):
    def hp(H1=A, H2=A, d=64, hd=256, chunk=16, B_=1):
        return lib.ttt_mlp_prefill_hist(A, A, A, A, A, A, A, A, A, H1, H2, B_, 1, 16, d, hd, chunk, 1, None)

    assert hp(H1=NULL) == T.TTT_ERR_INVALID_ARG
    assert hp(H2=MIS) == T.TTT_ERR_INVALID_ARG
    assert hp(d=128) == T.TTT_ERR_UNSUPPORTED
    assert hp(H1=NULL, H2=NULL, B_=0) == T.TTT_OK

    def bp(dW1T=A, dW10=A, chunk=16, d=64, hd=256, B_=1):
        return lib.ttt_mlp_prefill_backward(A, A, A, A, A, A, A, dW1T, A, A, A, A, A, dW10, A, B_, 1, 16, d, hd,
                                            chunk, 1, None)

    assert bp(dW10=NULL) == T.TTT_ERR_INVALID_ARG
    assert bp(dW1T=MIS) == T.TTT_ERR_INVALID_ARG
    assert bp(chunk=32, hd=64) == T.TTT_ERR_UNSUPPORTED  # the backward takes blocks of at most 16 tokens
    assert b"16" in lib.ttt_last_error()
    assert bp(d=48) == T.TTT_ERR_UNSUPPORTED
    assert bp(B_=0) == T.TTT_OK
