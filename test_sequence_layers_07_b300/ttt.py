"""Python binding of libttt.so (include/ttt.h): argument marshalling only.

The functions named like the C entry points (``ttt_linear_prefill``,
``ttt_mlp_prefill``, ``ttt_linear_decode_step``) take torch CUDA tensors,
check their dtype/shape/contiguity, pass raw device pointers and the current
CUDA stream to the library and raise :class:`TTTError` on a non-OK status.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback.  If libttt.so is missing, importing the library
raises immediately (build it with ``python -m test_sequence_layers_07_b300.build``).

The lower-case helpers (``linear_prefill`` ...) allocate the outputs with
torch and call the entry points above.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libttt.so")

TTT_OK, TTT_ERR_INVALID_ARG, TTT_ERR_UNSUPPORTED, TTT_ERR_CUDA, TTT_ERR_TIMEOUT = range(5)
TTT_F32, TTT_BF16 = 0, 1

EXPORTED = ("ttt_linear_prefill", "ttt_linear_prefill_workspace_size", "ttt_linear_prefill_ws",
            "ttt_linear_prefill_noalloc", "ttt_linear_momentum_prefill", "ttt_linear_prefill_hist",
            "ttt_mlp_prefill_hist", "ttt_mlp_prefill_backward", "ttt_linear_prefill_backward", "ttt_mlp_prefill",
            "ttt_linear_decode_step", "ttt_mlp_decode_step",
            "ttt_get_device_status", "ttt_selftest_wait_timeout", "ttt_status_string", "ttt_last_error", "ttt_version")


class TTTError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libttt.so once; raises FileNotFoundError if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise FileNotFoundError(
                    f"{path} not found: build the CUDA library with "
                    "`python -m test_sequence_layers_07_b300.build` (there is no fallback)")
            lib = ctypes.CDLL(path)
            vp, fp, i = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
            lib.ttt_linear_prefill.argtypes = [vp, vp, vp, fp, fp, vp, fp, i, i, i, i, i, i, vp]
            lib.ttt_linear_prefill_workspace_size.argtypes = [i, i, i, i, i, i]
            lib.ttt_linear_prefill_workspace_size.restype = ctypes.c_size_t
            lib.ttt_linear_prefill_ws.argtypes = [vp, vp, vp, fp, fp, vp, fp, i, i, i, i, i, i, vp, ctypes.c_size_t, vp]
            lib.ttt_linear_prefill_ws.restype = i
            lib.ttt_linear_prefill_noalloc.argtypes = [vp, vp, vp, fp, fp, vp, fp, i, i, i, i, i, i, vp]
            lib.ttt_linear_prefill_noalloc.restype = i
            lib.ttt_linear_momentum_prefill.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, fp, i, i, i, i, i,
                                                        ctypes.c_float, i, vp]
            lib.ttt_linear_momentum_prefill.restype = i
            lib.ttt_linear_prefill_hist.argtypes = [vp, vp, vp, fp, fp, vp, fp, fp, i, i, i, i, i, i, vp]
            lib.ttt_linear_prefill_backward.argtypes = [vp, vp, vp, fp, fp, vp, fp, vp, vp, vp, fp, fp,
                                                        i, i, i, i, i, i, vp]
            lib.ttt_mlp_prefill.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, fp, i, i, i, i, i, i, i, vp]
            lib.ttt_mlp_prefill_hist.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, fp, vp, vp, i, i, i, i, i, i, i, vp]
            lib.ttt_mlp_prefill_hist.restype = i
            lib.ttt_mlp_prefill_backward.argtypes = [vp, vp, vp, fp, vp, vp, vp, fp, fp, vp, vp, vp, fp, fp, fp,
                                                     i, i, i, i, i, i, i, vp]
            lib.ttt_mlp_prefill_backward.restype = i
            lib.ttt_linear_decode_step.argtypes = [vp, vp, vp, fp, fp, vp, i, i, i, i, vp]
            lib.ttt_mlp_decode_step.argtypes = [vp, vp, vp, fp, fp, fp, vp, i, i, i, i, i, vp]
            lib.ttt_get_device_status.argtypes = [vp]
            lib.ttt_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
            lib.ttt_selftest_wait_timeout.restype = i
            for f in (lib.ttt_linear_prefill, lib.ttt_linear_prefill_hist, lib.ttt_linear_prefill_backward,
                      lib.ttt_mlp_prefill, lib.ttt_linear_decode_step,
                      lib.ttt_mlp_decode_step, lib.ttt_get_device_status):
                f.restype = i
            lib.ttt_status_string.argtypes = [i]
            lib.ttt_status_string.restype = ctypes.c_char_p
            lib.ttt_last_error.argtypes = []
            lib.ttt_last_error.restype = ctypes.c_char_p
            lib.ttt_version.argtypes = []
            lib.ttt_version.restype = i
            _lib = lib
    return _lib


def _check(status: int):
    if status != TTT_OK:
        lib = load_library()
        msg = lib.ttt_last_error().decode() or lib.ttt_status_string(status).decode()
        raise TTTError(status, msg)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None, name: str, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _io_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return TTT_F32
    if t.dtype == torch.bfloat16:
        return TTT_BF16
    raise TypeError(f"Q/K/V must be float32 or bfloat16, got {t.dtype}")


def ttt_linear_prefill(Q, K, V, eta, W0, Z, W_out, chunk: int, stream=None) -> None:
    """TTT-Linear prefill into caller-allocated Z [B,H,T,d] and W_out [B,H,d,d] (may be W0)."""
    B, H, T, d = Q.shape
    dt = _io_dtype(Q)
    for name, t in (("K", K), ("V", V), ("Z", Z)):
        if t.shape != Q.shape or t.dtype != Q.dtype:
            raise ValueError(f"{name} must match Q in shape and dtype")
    if eta.shape != (B, H, T) or W0.shape != (B, H, d, d) or W_out.shape != (B, H, d, d):
        raise ValueError("eta must be [B,H,T] and W0/W_out [B,H,d,d]")
    st = load_library().ttt_linear_prefill(
        _ptr(Q, "Q"), _ptr(K, "K"), _ptr(V, "V"), _ptr(eta, "eta", torch.float32), _ptr(W0, "W0", torch.float32),
        _ptr(Z, "Z"), _ptr(W_out, "W_out", torch.float32), B, H, T, d, int(chunk), dt, _stream(stream))
    _check(st)


def ttt_linear_prefill_workspace_size(B: int, H: int, T: int, d: int, chunk: int, dtype: torch.dtype) -> int:
    """Bytes of scratch ttt_linear_prefill_ws needs for this shape (0: it runs the one-pass scan)."""
    dt = TTT_BF16 if dtype == torch.bfloat16 else TTT_F32
    return int(load_library().ttt_linear_prefill_workspace_size(B, H, T, d, int(chunk), dt))


def ttt_linear_prefill_ws(Q, K, V, eta, W0, Z, W_out, chunk: int, workspace, stream=None) -> None:
    """TTT-Linear prefill split along the sequence, with caller-owned scratch `workspace` (a CUDA
    tensor of at least ttt_linear_prefill_workspace_size bytes, or None when that size is 0)."""
    B, H, T, d = Q.shape
    dt = _io_dtype(Q)
    for name, t in (("K", K), ("V", V), ("Z", Z)):
        if t.shape != Q.shape or t.dtype != Q.dtype:
            raise ValueError(f"{name} must match Q in shape and dtype")
    if eta.shape != (B, H, T) or W0.shape != (B, H, d, d) or W_out.shape != (B, H, d, d):
        raise ValueError("eta must be [B,H,T] and W0/W_out [B,H,d,d]")
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load_library().ttt_linear_prefill_ws(
        _ptr(Q, "Q"), _ptr(K, "K"), _ptr(V, "V"), _ptr(eta, "eta", torch.float32), _ptr(W0, "W0", torch.float32),
        _ptr(Z, "Z"), _ptr(W_out, "W_out", torch.float32), B, H, T, d, int(chunk), dt,
        _ptr(workspace, "workspace"), nbytes, _stream(stream))
    _check(st)


def ttt_linear_prefill_noalloc(Q, K, V, eta, W0, Z, W_out, chunk: int, stream=None) -> None:
    """The split TTT-Linear prefill with the library's built-in scratch (no workspace argument, nothing
    allocated): for callers that cannot allocate device memory when they run the scan."""
    B, H, T, d = Q.shape
    dt = _io_dtype(Q)
    for name, t in (("K", K), ("V", V), ("Z", Z)):
        if t.shape != Q.shape or t.dtype != Q.dtype:
            raise ValueError(f"{name} must match Q in shape and dtype")
    if eta.shape != (B, H, T) or W0.shape != (B, H, d, d) or W_out.shape != (B, H, d, d):
        raise ValueError("eta must be [B,H,T] and W0/W_out [B,H,d,d]")
    st = load_library().ttt_linear_prefill_noalloc(
        _ptr(Q, "Q"), _ptr(K, "K"), _ptr(V, "V"), _ptr(eta, "eta", torch.float32), _ptr(W0, "W0", torch.float32),
        _ptr(Z, "Z"), _ptr(W_out, "W_out", torch.float32), B, H, T, d, int(chunk), dt, _stream(stream))
    _check(st)


def ttt_linear_momentum_prefill(Q, K, V, eta, W0, M0, Z, W_out, M_out, chunk: int, beta: float,
                                stream=None) -> None:
    """TTT-Linear prefill with momentum: M0 [B,H,d,d] fp32 or None (zero), outputs Z, W_out and
    M_out (each may alias its input state)."""
    B, H, T, d = Q.shape
    dt = _io_dtype(Q)
    for name, t in (("K", K), ("V", V), ("Z", Z)):
        if t.shape != Q.shape or t.dtype != Q.dtype:
            raise ValueError(f"{name} must match Q in shape and dtype")
    for name, t in (("W0", W0), ("W_out", W_out), ("M_out", M_out), ("M0", M0)):
        if t is not None and t.shape != (B, H, d, d):
            raise ValueError(f"{name} must be [B,H,d,d]")
    if eta.shape != (B, H, T):
        raise ValueError("eta must be [B,H,T]")
    st = load_library().ttt_linear_momentum_prefill(
        _ptr(Q, "Q"), _ptr(K, "K"), _ptr(V, "V"), _ptr(eta, "eta", torch.float32), _ptr(W0, "W0", torch.float32),
        _ptr(M0, "M0", torch.float32), _ptr(Z, "Z"), _ptr(W_out, "W_out", torch.float32),
        _ptr(M_out, "M_out", torch.float32), B, H, T, d, int(chunk), float(beta), dt, _stream(stream))
    _check(st)


def ttt_linear_prefill_hist(Q, K, V, eta, W0, Z, W_out, W_hist, chunk: int, stream=None) -> None:
    """TTT-Linear prefill that also writes the state at the start of every block into
    W_hist [B,H,ceil(T/chunk),d,d] (the input of the backward), in the dtype of Q: fp32, or for
    bf16 inputs the state rounded to bf16."""
    B, H, T, d = Q.shape
    dt = _io_dtype(Q)
    for name, t in (("K", K), ("V", V), ("Z", Z)):
        if t.shape != Q.shape or t.dtype != Q.dtype:
            raise ValueError(f"{name} must match Q in shape and dtype")
    nblk = -(-T // int(chunk)) if chunk > 0 else 0
    if eta.shape != (B, H, T) or W0.shape != (B, H, d, d) or W_out.shape != (B, H, d, d):
        raise ValueError("eta must be [B,H,T] and W0/W_out [B,H,d,d]")
    if W_hist.shape != (B, H, nblk, d, d):
        raise ValueError("W_hist must be [B,H,ceil(T/chunk),d,d]")
    st = load_library().ttt_linear_prefill_hist(
        _ptr(Q, "Q"), _ptr(K, "K"), _ptr(V, "V"), _ptr(eta, "eta", torch.float32), _ptr(W0, "W0", torch.float32),
        _ptr(Z, "Z"), _ptr(W_out, "W_out", torch.float32), _ptr(W_hist, "W_hist", Q.dtype),
        B, H, T, d, int(chunk), dt, _stream(stream))
    _check(st)


def ttt_linear_prefill_backward(Q, K, V, eta, W_hist, dZ, dW_T, dQ, dK, dV, deta, dW0, chunk: int,
                                stream=None) -> None:
    """Gradient of the TTT-Linear prefill: dQ, dK, dV [B,H,T,d] (dtype of Q), deta [B,H,T] and
    dW0 [B,H,d,d] (fp32) from dZ and dW_T (None: zero)."""
    B, H, T, d = Q.shape
    dt = _io_dtype(Q)
    for name, t in (("K", K), ("V", V), ("dZ", dZ), ("dQ", dQ), ("dK", dK), ("dV", dV)):
        if t.shape != Q.shape or t.dtype != Q.dtype:
            raise ValueError(f"{name} must match Q in shape and dtype")
    nblk = -(-T // int(chunk)) if chunk > 0 else 0
    if eta.shape != (B, H, T) or deta.shape != (B, H, T) or dW0.shape != (B, H, d, d):
        raise ValueError("eta/deta must be [B,H,T] and dW0 [B,H,d,d]")
    if W_hist.shape != (B, H, nblk, d, d) or (dW_T is not None and dW_T.shape != (B, H, d, d)):
        raise ValueError("W_hist must be [B,H,ceil(T/chunk),d,d] and dW_T [B,H,d,d]")
    st = load_library().ttt_linear_prefill_backward(
        _ptr(Q, "Q"), _ptr(K, "K"), _ptr(V, "V"), _ptr(eta, "eta", torch.float32),
        _ptr(W_hist, "W_hist", Q.dtype), _ptr(dZ, "dZ"), _ptr(dW_T, "dW_T", torch.float32), _ptr(dQ, "dQ"),
        _ptr(dK, "dK"), _ptr(dV, "dV"), _ptr(deta, "deta", torch.float32), _ptr(dW0, "dW0", torch.float32),
        B, H, T, d, int(chunk), dt, _stream(stream))
    _check(st)


def ttt_mlp_prefill(Q, K, V, eta, W1_0, W2_0, Z, W1_out, W2_out, chunk: int, stream=None) -> None:
    """TTT-MLP prefill into caller-allocated Z, W1_out [B,H,d,hidden], W2_out [B,H,hidden,d]."""
    B, H, T, d = Q.shape
    hidden = W1_0.shape[-1]
    dt = _io_dtype(Q)
    for name, t in (("K", K), ("V", V), ("Z", Z)):
        if t.shape != Q.shape or t.dtype != Q.dtype:
            raise ValueError(f"{name} must match Q in shape and dtype")
    if eta.shape != (B, H, T) or W1_0.shape != (B, H, d, hidden) or W2_0.shape != (B, H, hidden, d):
        raise ValueError("eta must be [B,H,T], W1 [B,H,d,hidden], W2 [B,H,hidden,d]")
    if W1_out.shape != W1_0.shape or W2_out.shape != W2_0.shape:
        raise ValueError("output weights must match the input weights' shapes")
    st = load_library().ttt_mlp_prefill(
        _ptr(Q, "Q"), _ptr(K, "K"), _ptr(V, "V"), _ptr(eta, "eta", torch.float32),
        _ptr(W1_0, "W1_0", torch.float32), _ptr(W2_0, "W2_0", torch.float32), _ptr(Z, "Z"),
        _ptr(W1_out, "W1_out", torch.float32), _ptr(W2_out, "W2_out", torch.float32),
        B, H, T, d, hidden, int(chunk), dt, _stream(stream))
    _check(st)


def ttt_mlp_prefill_hist(Q, K, V, eta, W1_0, W2_0, Z, W1_out, W2_out, W1_hist, W2_hist, chunk: int,
                         stream=None) -> None:
    """TTT-MLP prefill that also writes the block-start states into W1_hist [B,H,nblk,d,hidden] and
    W2_hist [B,H,nblk,hidden,d] (dtype of Q)."""
    B, H, T, d = Q.shape
    hd = W1_0.shape[-1]
    dt = _io_dtype(Q)
    nblk = -(-T // int(chunk))
    if W1_hist.shape != (B, H, nblk, d, hd) or W2_hist.shape != (B, H, nblk, hd, d):
        raise ValueError("W1_hist must be [B,H,nblk,d,hidden] and W2_hist [B,H,nblk,hidden,d]")
    if W1_hist.dtype != Q.dtype or W2_hist.dtype != Q.dtype:
        raise TypeError("W1_hist / W2_hist must have the dtype of Q")
    st = load_library().ttt_mlp_prefill_hist(
        _ptr(Q, "Q"), _ptr(K, "K"), _ptr(V, "V"), _ptr(eta, "eta", torch.float32), _ptr(W1_0, "W1_0", torch.float32),
        _ptr(W2_0, "W2_0", torch.float32), _ptr(Z, "Z"), _ptr(W1_out, "W1_out", torch.float32),
        _ptr(W2_out, "W2_out", torch.float32), _ptr(W1_hist, "W1_hist"), _ptr(W2_hist, "W2_hist"), B, H, T, d, hd,
        int(chunk), dt, _stream(stream))
    _check(st)


def ttt_mlp_prefill_backward(Q, K, V, eta, W1_hist, W2_hist, dZ, dW1_T, dW2_T, dQ, dK, dV, deta, dW1_0, dW2_0,
                             chunk: int, stream=None) -> None:
    """Gradient of the TTT-MLP prefill into caller-allocated dQ, dK, dV, deta, dW1_0, dW2_0."""
    B, H, T, d = Q.shape
    hd = W1_hist.shape[-1]
    dt = _io_dtype(Q)
    st = load_library().ttt_mlp_prefill_backward(
        _ptr(Q, "Q"), _ptr(K, "K"), _ptr(V, "V"), _ptr(eta, "eta", torch.float32), _ptr(W1_hist, "W1_hist"),
        _ptr(W2_hist, "W2_hist"), _ptr(dZ, "dZ"), _ptr(dW1_T, "dW1_T", torch.float32),
        _ptr(dW2_T, "dW2_T", torch.float32), _ptr(dQ, "dQ"), _ptr(dK, "dK"), _ptr(dV, "dV"),
        _ptr(deta, "deta", torch.float32), _ptr(dW1_0, "dW1_0", torch.float32), _ptr(dW2_0, "dW2_0", torch.float32),
        B, H, T, d, hd, int(chunk), dt, _stream(stream))
    _check(st)


def ttt_linear_decode_step(q, k, v, eta, W, z, stream=None) -> None:
    """One online TTT-Linear step; W [B,H,d,d] fp32 is updated in place, z written."""
    B, H, d = q.shape
    dt = _io_dtype(q)
    for name, t in (("k", k), ("v", v), ("z", z)):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must match q in shape and dtype")
    if eta.shape != (B, H) or W.shape != (B, H, d, d):
        raise ValueError("eta must be [B,H] and W [B,H,d,d]")
    st = load_library().ttt_linear_decode_step(
        _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(eta, "eta", torch.float32), _ptr(W, "W", torch.float32),
        _ptr(z, "z"), B, H, d, dt, _stream(stream))
    _check(st)


def ttt_mlp_decode_step(q, k, v, eta, W1, W2, z, stream=None) -> None:
    """One online TTT-MLP step; W1 [B,H,d,hidden] and W2 [B,H,hidden,d] (fp32) updated in place, z written."""
    B, H, d = q.shape
    hidden = W1.shape[-1]
    dt = _io_dtype(q)
    for name, t in (("k", k), ("v", v), ("z", z)):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must match q in shape and dtype")
    if eta.shape != (B, H) or W1.shape != (B, H, d, hidden) or W2.shape != (B, H, hidden, d):
        raise ValueError("eta must be [B,H], W1 [B,H,d,hidden] and W2 [B,H,hidden,d]")
    st = load_library().ttt_mlp_decode_step(
        _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(eta, "eta", torch.float32), _ptr(W1, "W1", torch.float32),
        _ptr(W2, "W2", torch.float32), _ptr(z, "z"), B, H, d, hidden, dt, _stream(stream))
    _check(st)


def ttt_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    """Launches the device-side bounded-wait self-test (records TTT_ERR_TIMEOUT after `limit_ns`)."""
    _check(load_library().ttt_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def ttt_get_device_status(stream=None) -> int:
    """Reads and clears the device status word (synchronises the stream); returns the status code."""
    return load_library().ttt_get_device_status(_stream(stream))


# ---------------------------------------------------------------- helpers

def linear_prefill(Q, K, V, eta, W0, chunk: int, stream=None):
    """Returns (Z, W_final) for a TTT-Linear prefill, outputs allocated by torch."""
    Z = torch.empty_like(Q)
    W = torch.empty_like(W0)
    ttt_linear_prefill(Q, K, V, eta, W0, Z, W, chunk, stream)
    return Z, W


def linear_workspace(Q, chunk: int):
    """A scratch buffer for ttt_linear_prefill_ws on Q's shape (None when none is needed)."""
    B, H, T, d = Q.shape
    n = ttt_linear_prefill_workspace_size(B, H, T, d, chunk, Q.dtype)
    return torch.empty(n // 4, dtype=torch.float32, device=Q.device) if n else None


def linear_prefill_ws(Q, K, V, eta, W0, chunk: int, workspace=None, stream=None):
    """Returns (Z, W_final) for the TTT-Linear prefill split along the sequence (scratch allocated by
    torch when not given)."""
    if workspace is None:
        workspace = linear_workspace(Q, chunk)
    Z = torch.empty_like(Q)
    W = torch.empty_like(W0)
    ttt_linear_prefill_ws(Q, K, V, eta, W0, Z, W, chunk, workspace, stream)
    return Z, W


def linear_momentum_prefill(Q, K, V, eta, W0, M0, chunk: int, beta: float, stream=None):
    """Returns (Z, W_final, M_final) for the TTT-Linear prefill with momentum (M0 None: zero)."""
    Z = torch.empty_like(Q)
    W = torch.empty_like(W0)
    M = torch.empty_like(W0)
    ttt_linear_momentum_prefill(Q, K, V, eta, W0, M0, Z, W, M, chunk, beta, stream)
    return Z, W, M


def linear_prefill_hist(Q, K, V, eta, W0, chunk: int, stream=None):
    """Returns (Z, W_final, W_hist) for a TTT-Linear prefill that records the block-start states."""
    B, H, T, d = Q.shape
    Z = torch.empty_like(Q)
    W = torch.empty_like(W0)
    Wh = torch.empty((B, H, -(-T // int(chunk)), d, d), dtype=Q.dtype, device=Q.device)
    ttt_linear_prefill_hist(Q, K, V, eta, W0, Z, W, Wh, chunk, stream)
    return Z, W, Wh


def linear_prefill_backward(Q, K, V, eta, W_hist, dZ, dW_T, chunk: int, stream=None):
    """Returns (dQ, dK, dV, deta, dW0) of the TTT-Linear prefill."""
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(Q), torch.empty_like(Q)
    deta = torch.empty_like(eta)
    dW0 = torch.empty(W_hist.shape[:2] + W_hist.shape[3:], dtype=torch.float32, device=Q.device)
    ttt_linear_prefill_backward(Q, K, V, eta, W_hist, dZ, dW_T, dQ, dK, dV, deta, dW0, chunk, stream)
    return dQ, dK, dV, deta, dW0


def mlp_prefill(Q, K, V, eta, W1, W2, chunk: int, stream=None):
    """Returns (Z, W1_final, W2_final) for a TTT-MLP prefill."""
    Z = torch.empty_like(Q)
    W1o = torch.empty_like(W1)
    W2o = torch.empty_like(W2)
    ttt_mlp_prefill(Q, K, V, eta, W1, W2, Z, W1o, W2o, chunk, stream)
    return Z, W1o, W2o


def mlp_prefill_hist(Q, K, V, eta, W1, W2, chunk: int, stream=None):
    """Returns (Z, W1_final, W2_final, W1_hist, W2_hist) for a TTT-MLP prefill that records the
    block-start states."""
    B, H, T, d = Q.shape
    hd = W1.shape[-1]
    nblk = -(-T // int(chunk))
    Z, W1o, W2o = torch.empty_like(Q), torch.empty_like(W1), torch.empty_like(W2)
    H1 = torch.empty((B, H, nblk, d, hd), dtype=Q.dtype, device=Q.device)
    H2 = torch.empty((B, H, nblk, hd, d), dtype=Q.dtype, device=Q.device)
    ttt_mlp_prefill_hist(Q, K, V, eta, W1, W2, Z, W1o, W2o, H1, H2, chunk, stream)
    return Z, W1o, W2o, H1, H2


def mlp_prefill_backward(Q, K, V, eta, W1_hist, W2_hist, dZ, dW1_T, dW2_T, chunk: int, stream=None):
    """Returns (dQ, dK, dV, deta, dW1_0, dW2_0) of the TTT-MLP prefill."""
    B, H, T, d = Q.shape
    hd = W1_hist.shape[-1]
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(Q), torch.empty_like(Q)
    deta = torch.empty_like(eta)
    dW1 = torch.empty((B, H, d, hd), dtype=torch.float32, device=Q.device)
    dW2 = torch.empty((B, H, hd, d), dtype=torch.float32, device=Q.device)
    ttt_mlp_prefill_backward(Q, K, V, eta, W1_hist, W2_hist, dZ, dW1_T, dW2_T, dQ, dK, dV, deta, dW1, dW2, chunk,
                             stream)
    return dQ, dK, dV, deta, dW1, dW2


def mlp_decode_step(q, k, v, eta, W1, W2, stream=None):
    """Returns z; W1 and W2 are updated in place."""
    z = torch.empty_like(q)
    ttt_mlp_decode_step(q, k, v, eta, W1, W2, z, stream)
    return z


def linear_decode_step(q, k, v, eta, W, stream=None):
    """Returns z; W is updated in place."""
    z = torch.empty_like(q)
    ttt_linear_decode_step(q, k, v, eta, W, z, stream)
    return z
