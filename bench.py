#!/usr/bin/env python3
"""Throughput of the TTT inner-loop scan library on one B300 (or N, one process each).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--rows all|none]

A step is one TTT-Linear prefill over the headline workload (B=8, H=12,
d=64, T=2048, chunk 16, bf16 Q/K/V/Z, fp32 state): the §-named "linear
prefill" configuration the metric is quoted on.  Four copies of the inputs
(4 x 105 MB > 126 MB L2) rotate from step to step so every step reads from HBM.
The JSON line printed by rank 0 carries the headline value (tokens/s over all
ranks), its roofline fraction, the clocks seen during the timed region, the
end-to-end number through the public API with host buffers, the oracle's CPU
baseline, and under "rows" the other workloads (TTT-MLP prefill, the
long-context chunk sweep, the TTT-Linear and TTT-MLP decode steps), each timed
the same way.

--impl reference times the fp64 CPU oracle (test infrastructure) on the host
cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from test_sequence_layers_07_b300 import workloads as WL  # noqa: E402

METRIC = "TTT-Linear/MLP prefill tokens/s & % roofline; decode tokens/s & HBM GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# the B300's rated figures: HBM3e bandwidth and dense bf16 tensor throughput
RATED_PEAKS = {"hbm_gbs": 7700.0, "bf16_tflops": 2250.0}
# fp32 FMA peak of the SIMT pipes: 148 SMs x 128 FMA lanes x 2 FLOP x 2.032 GHz (the maximum SM clock), the
# ceiling of the kernels that run their contractions as plain fp32 multiply-adds
FP32_ALU_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12
NROT = 4  # rotating input copies for the L2-sized workloads


# ------------------------------------------------------------------ helpers

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def rated_roof(nbytes, flops):
    """Roofline time (s) against the rated peaks instead of the measured ones."""
    return max(nbytes / (RATED_PEAKS["hbm_gbs"] * 1e9), flops / (RATED_PEAKS["bf16_tflops"] * 1e12))


def linear_bytes(B, H, T, d, elt=2):
    """Algorithmic HBM bytes of one TTT-Linear prefill: Q,K,V read + Z written, eta, W0 read + W written."""
    return 4 * B * H * T * d * elt + 4 * B * H * T + 2 * B * H * d * d * 4


def linear_flops(B, H, T, d, b):
    """Dual-form FLOPs: Q W0, K W0, K^T E (2d^2 each per token) + causal Q K^T and A E ((b+1)d each)."""
    return B * H * T * (6 * d * d + 2 * (b + 1) * d)


def mlp_flops(B, H, T, d, hd, b):
    return B * H * T * (14 * d * hd + 2 * (b + 1) * (d + hd))


def mlp_bytes(B, H, T, d, hd, elt=2):
    return 4 * B * H * T * d * elt + 4 * B * H * T + 2 * 2 * B * H * d * hd * 4


def decode_bytes(B, H, d, elt=2):
    """Per step: state read + written once, q,k,v read, z written, eta read."""
    return 2 * B * H * d * d * 4 + 4 * B * H * d * elt + 4 * B * H


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "test_sequence_layers_07_b300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key, src_files):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current source."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d or d.get("source_sha") != kernel_source_hash(src_files):
        return None
    return d.get("dram_bytes_per_launch")


class _Nvml:
    """Minimal ctypes binding of libnvidia-ml (clock and clock-event-reason queries only)."""

    def __init__(self):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")

    def handle(self, pci_bus_id: str):
        h = self.c.c_void_p()
        r = self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), self.c.byref(h))
        if r != 0:
            r = self.lib.nvmlDeviceGetHandleByIndex_v2(0, self.c.byref(h))
        if r != 0:
            raise RuntimeError(f"nvml handle lookup failed ({r})")
        return h

    def clock(self, h, max_=False):
        v = self.c.c_uint()
        f = self.lib.nvmlDeviceGetMaxClockInfo if max_ else self.lib.nvmlDeviceGetClockInfo
        if f(h, 1, self.c.byref(v)) != 0:  # 1 = NVML_CLOCK_SM
            raise RuntimeError("clock query failed")
        return v.value

    def reasons(self, h):
        v = self.c.c_ulonglong()
        if self.lib.nvmlDeviceGetCurrentClocksEventReasons(h, self.c.byref(v)) != 0:
            raise RuntimeError("reason query failed")
        return v.value


class ClockSampler:
    """Samples SM clock and clock-event reasons (NVML through ctypes) while the timed region runs."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting", 0x1: "gpu_idle",
               0x10: "sync_boost"}

    def __init__(self, device=0, interval=0.002):
        self.interval = interval
        self.samples, self.reasons = [], set()
        self.max_mhz = None
        self._stop = threading.Event()
        self._err = None
        self._nv = None
        try:
            self._nv = _Nvml()
            props = torch.cuda.get_device_properties(device)
            bus = "%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
            self._h = self._nv.handle(bus)
            self.max_mhz = self._nv.clock(self._h, max_=True)
        except Exception as e:
            self._nv = None
            self._err = f"nvml: {e!r}"

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self._nv.clock(self._h))
                r = self._nv.reasons(self._h)
                for bit, name in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(self.interval)

    def __enter__(self):
        if self._nv is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self._nv is not None:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "note": self._err or "no samples in the timed region"}
        reasons = sorted(self.reasons - {"gpu_idle"})
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples)}


def dist_setup(gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Max of a per-rank scalar (host-side bookkeeping; no data-path collective)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# Timed regions replay the K steps as one CUDA graph (the launches the steps make, captured in order with
# their rotating inputs), so the device time is measured without the host's per-call launch work in the
# way; --eager times per-call launches instead.
GRAPH = True


def timed_loop(fn, steps, warmup, world, stream=None, sampler=None, min_warm_s=0.3, graph=None):
    """Runs `fn(i)` warmup times untimed, then `steps` times between two barriers + syncs.

    Warm-up runs at least `warmup` steps and at least `min_warm_s` seconds (so the
    clocks have ramped up).  Returns (ms_per_step over the whole region, max over
    ranks; mean per-launch ms: from per-call CUDA events on the launching stream when
    launching eagerly, the region divided by the steps when replaying a graph).  `graph` (default:
    the module's GRAPH) is False for steps that are graph replays themselves.
    """
    stream = stream or torch.cuda.current_stream()
    t_start = time.perf_counter()
    i = 0
    while i < warmup or time.perf_counter() - t_start < min_warm_s:
        fn(i)
        i += 1
        if i % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    warmup = i
    if GRAPH if graph is None else graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for j in range(steps):
                fn(warmup + j)
        torch.cuda.synchronize()
        g.replay()  # one untimed replay: the graph's first launch uploads it
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        ctx = sampler if sampler is not None else _Null()
        with ctx:
            t0.record(stream)
            g.replay()
            t1.record(stream)
            torch.cuda.synchronize()
        barrier(world)
        total = t0.elapsed_time(t1)
        del g
        return max_over_ranks(total / steps, world), total / steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        t0.record(stream)
        for i in range(steps):
            ev[i][0].record(stream)
            fn(warmup + i)
            ev[i][1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    total = t0.elapsed_time(t1)
    per_launch = sum(a.elapsed_time(b) for a, b in ev) / steps
    return max_over_ranks(total / steps, world), per_launch


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


# ---------------------------------------------------------------- our arm

def rotating_copies(x: dict, n: int) -> list:
    base = {k: v.cuda() for k, v in x.items()}
    return [base] + [{k: v.clone() for k, v in base.items()} for _ in range(n - 1)]


def linear_launches(T_mod, w, chunk, split):
    """Kernel launches of one prefill call: the split path runs maps, combine and scan (3) when its
    workspace is non-empty, the one-pass path 1."""
    if not split:
        return 1
    n = T_mod.ttt_linear_prefill_workspace_size(w.B, w.H, w.T, w.d, chunk, WL.torch_dtype(w.dtype))
    return 3 if n else 1


def segments_of(ws, w):
    """Segment count of a split prefill from its workspace size (B*H*(3S-2)*d*d fp32 words)."""
    if ws is None:
        return 1
    return (ws.numel() // (w.B * w.H * w.d * w.d) + 2) // 3


def bench_linear(T_mod, w, chunk, steps, warmup, world, peaks, sampler=None, nrot=NROT, split=False):
    """One TTT-Linear prefill per step: split along the sequence (ttt_linear_prefill_ws, scratch
    allocated once, outside the timed region) or the one-pass scan (ttt_linear_prefill)."""
    x = WL.workload_inputs(w)
    sets = rotating_copies(x, nrot)
    outs = [(torch.empty_like(s["Q"]), torch.empty_like(s["W0"])) for s in sets]
    ws = T_mod.linear_workspace(sets[0]["Q"], chunk) if split else None

    def step(i):
        s, (Z, W) = sets[i % nrot], outs[i % nrot]
        if split:
            T_mod.ttt_linear_prefill_ws(s["Q"], s["K"], s["V"], s["eta"], s["W0"], Z, W, chunk, ws)
        else:
            T_mod.ttt_linear_prefill(s["Q"], s["K"], s["V"], s["eta"], s["W0"], Z, W, chunk)

    ms, ms_launch = timed_loop(step, steps, warmup, world, sampler=sampler)
    toks = w.B * w.T
    nbytes = linear_bytes(w.B, w.H, w.T, w.d)
    flops = linear_flops(w.B, w.H, w.T, w.d, chunk)
    t_roof = max(nbytes / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
    nseg = segments_of(ws, w) if split else 1
    del sets, outs, ws
    return {"tokens_per_s": toks / (ms * 1e-3), "ms_per_step": ms, "ms_per_launch": ms_launch,
            "path": "split along the sequence" if split else "one pass", "segments": nseg,
            "kernel_launches_per_call": linear_launches(T_mod, w, chunk, split),
            "bytes_per_launch": nbytes, "flops_per_launch": flops,
            "achieved_gbs": nbytes / (ms_launch * 1e-3) / 1e9, "roofline_us": t_roof * 1e6,
            "frac": t_roof / (ms_launch * 1e-3), "bound": "hbm",
            "frac_of_rated": rated_roof(nbytes, flops) / (ms_launch * 1e-3)}


def bench_mlp(T_mod, w, steps, warmup, world, peaks):
    x = WL.workload_inputs(w)
    sets = rotating_copies(x, NROT)
    outs = [(torch.empty_like(s["Q"]), torch.empty_like(s["W1"]), torch.empty_like(s["W2"])) for s in sets]

    def step(i):
        s, (Z, W1, W2) = sets[i % NROT], outs[i % NROT]
        T_mod.ttt_mlp_prefill(s["Q"], s["K"], s["V"], s["eta"], s["W1"], s["W2"], Z, W1, W2, w.chunk)

    ms, ms_launch = timed_loop(step, steps, warmup, world)
    flops = mlp_flops(w.B, w.H, w.T, w.d, w.hidden, w.chunk)
    nbytes = mlp_bytes(w.B, w.H, w.T, w.d, w.hidden)
    t_tensor = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    del sets, outs
    return {"tokens_per_s": w.B * w.T / (ms * 1e-3), "ms_per_step": ms, "ms_per_launch": ms_launch,
            "flops_per_launch": flops, "bytes_per_launch": nbytes,
            "achieved_tflops": flops / (ms_launch * 1e-3) / 1e12, "roofline_us": max(t_tensor, t_hbm) * 1e6,
            "frac": max(t_tensor, t_hbm) / (ms_launch * 1e-3), "bound": "tensor" if t_tensor > t_hbm else "hbm",
            "frac_of_rated": rated_roof(nbytes, flops) / (ms_launch * 1e-3)}


def momentum_bytes(B, H, T, d, elt=2):
    """Momentum prefill: the plain prefill's bytes plus the fp32 momentum read and written once."""
    return linear_bytes(B, H, T, d, elt) + 2 * B * H * d * d * 4


def momentum_flops(B, H, T, d, b):
    """Q W, K W, Q M and the two rank updates (W and M), 2 d^2 each per token, plus the causal
    products ((b + 1) d each, two)."""
    return B * H * T * (10 * d * d + 2 * (b + 1) * d)


def bench_momentum(T_mod, w, beta, steps, warmup, world, peaks, nrot=2):
    x = WL.workload_inputs(w)
    rng = torch.Generator().manual_seed(w.seed + 200)
    x["M0"] = (torch.randn(x["W0"].shape, generator=rng) * 0.02).float()
    sets = rotating_copies(x, nrot)
    outs = [(torch.empty_like(s["Q"]), torch.empty_like(s["W0"]), torch.empty_like(s["W0"])) for s in sets]

    def step(i):
        s, (Z, W, M) = sets[i % nrot], outs[i % nrot]
        T_mod.ttt_linear_momentum_prefill(s["Q"], s["K"], s["V"], s["eta"], s["W0"], s["M0"], Z, W, M, w.chunk, beta)

    ms, ms_launch = timed_loop(step, steps, warmup, world)
    # the library's choice for this shape (include/ttt.h)
    mma = (w.dtype == "bf16" and w.d == 64 and w.chunk == 16 and w.T % 16 == 0
           and os.environ.get("TTT_LINEAR_MOMENTUM_KERNEL") != "simt")
    kernel = "warp-level MMA, bf16 operands" if mma else "SIMT fp32 (generic)"
    nbytes = momentum_bytes(w.B, w.H, w.T, w.d)
    flops = momentum_flops(w.B, w.H, w.T, w.d, w.chunk)
    t_roof = max(nbytes / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
    del sets, outs
    return {"tokens_per_s": w.B * w.T / (ms * 1e-3), "ms_per_step": ms, "ms_per_launch": ms_launch, "beta": beta,
            "bytes_per_launch": nbytes, "flops_per_launch": flops, "roofline_us": t_roof * 1e6,
            "frac": t_roof / (ms_launch * 1e-3), "frac_of_rated": rated_roof(nbytes, flops) / (ms_launch * 1e-3),
            "bound": "hbm" if nbytes / (peaks["hbm_gbs"] * 1e9) > flops / (peaks["bf16_tflops"] * 1e12) else "tensor",
            "kernel": kernel}


def backward_bytes(B, H, T, d, chunk, elt=2):
    """Backward pass: Q,K,V,dZ read and dQ,dK,dV written (elt bytes each), eta read and deta written,
    the block-start states read once (elt bytes each: recorded in the dtype of Q), dW_T read and dW0
    written (fp32)."""
    nblk = -(-T // chunk)
    return B * H * (T * (7 * d * elt + 8) + nblk * d * d * elt + 2 * d * d * 4)


def backward_flops(B, H, T, d, chunk):
    """Per head-token: E, K dW', dQ's dZ W^T, dK's two d x d products and the two rank updates of dW
    (2 d^2 each, 7 in all) plus the causal score products S, dA, dE, dQ, dK ((b + 1) d each, 5)."""
    return B * H * T * (14 * d * d + 5 * (chunk + 1) * d)


def bench_backward(T_mod, w, steps, warmup, world, peaks, nrot=2):
    """Training step of the headline shape: the forward that records the block-start states, then
    the backward; both timed, each on its own launches."""
    x = WL.workload_inputs(w)
    g = WL.backward_inputs(w.B, w.H, w.T, w.d, seed=w.seed + 100, dtype=w.dtype)
    sets = rotating_copies({**x, "dZ": g["dZ"], "dWT": g["dWT"]}, nrot)
    nblk = -(-w.T // w.chunk)
    hist = [torch.empty((w.B, w.H, nblk, w.d, w.d), dtype=sets[0]["Q"].dtype, device="cuda") for _ in range(nrot)]
    fwd_out = [(torch.empty_like(s["Q"]), torch.empty_like(s["W0"])) for s in sets]
    bwd_out = [(torch.empty_like(s["Q"]), torch.empty_like(s["Q"]), torch.empty_like(s["Q"]),
                torch.empty_like(s["eta"]), torch.empty_like(s["W0"])) for s in sets]

    def fwd(i):
        s, (Z, W) = sets[i % nrot], fwd_out[i % nrot]
        T_mod.ttt_linear_prefill_hist(s["Q"], s["K"], s["V"], s["eta"], s["W0"], Z, W, hist[i % nrot], w.chunk)

    def bwd(i):
        s, o = sets[i % nrot], bwd_out[i % nrot]
        T_mod.ttt_linear_prefill_backward(s["Q"], s["K"], s["V"], s["eta"], hist[i % nrot], s["dZ"], s["dWT"],
                                          *o, w.chunk)

    for i in range(nrot):
        fwd(i)
    ms_f, ms_f_launch = timed_loop(fwd, steps, warmup, world)
    ms_b, ms_b_launch = timed_loop(bwd, steps, warmup, world)
    nbytes = backward_bytes(w.B, w.H, w.T, w.d, w.chunk)
    flops = backward_flops(w.B, w.H, w.T, w.d, w.chunk)
    t_roof = max(nbytes / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
    del sets, hist, fwd_out, bwd_out
    return {"tokens_per_s": w.B * w.T / ((ms_f + ms_b) * 1e-3), "ms_per_step": ms_f + ms_b,
            "forward_hist_ms_per_launch": ms_f_launch, "backward_ms_per_launch": ms_b_launch,
            "backward_bytes_per_launch": nbytes, "backward_flops_per_launch": flops,
            "backward_roofline_us": t_roof * 1e6, "backward_frac": t_roof / (ms_b_launch * 1e-3),
            "backward_frac_of_rated": rated_roof(nbytes, flops) / (ms_b_launch * 1e-3),
            "bound": "hbm" if nbytes / (peaks["hbm_gbs"] * 1e9) > flops / (peaks["bf16_tflops"] * 1e12) else "tensor"}


def mlp_backward_bytes(B, H, T, d, hd, chunk, elt=2):
    """TTT-MLP backward: Q, K, V, dZ read and dQ, dK, dV written (elt bytes each), eta read and deta
    written, the recorded W1, W2 of every block read once (elt bytes each), dW_T read and dW0 written
    (fp32, both layers)."""
    nblk = -(-T // chunk)
    return B * H * (T * (7 * d * elt + 8) + nblk * 2 * d * hd * elt + 2 * 2 * d * hd * 4)


def mlp_backward_flops(B, H, T, d, hd, chunk):
    """Per head-token: the block's forward at its start state (Zk, Zq, E2, Gk: 4 products) and the
    backward's products over d x hidden (dHk, dE1 from the state gradients, Hk dW2', E1 dW1'^T,
    dZ W2^T, dZq W1^T, dGk W2, dE2 W2^T, dZk W1^T, and the five rank updates of dW1, dW2), 2 d h each
    (18 in all), plus the causal score products ((b + 1)(d + h) each, six)."""
    return B * H * T * (36 * d * hd + 6 * (chunk + 1) * (d + hd))


def bench_mlp_backward(T_mod, w, steps, warmup, world, peaks, nrot=2):
    """Training step of the TTT-MLP workload shape: the forward that records the block-start states,
    then the backward; each timed on its own launches."""
    x = WL.workload_inputs(w)
    rng = torch.Generator().manual_seed(w.seed + 100)
    g = {"dZ": (torch.randn(x["Q"].shape, generator=rng) / w.d ** 0.5).to(x["Q"].dtype),
         "dW1T": torch.randn(x["W1"].shape, generator=rng) / w.d ** 0.5,
         "dW2T": torch.randn(x["W2"].shape, generator=rng) / w.d ** 0.5}
    sets = rotating_copies({**x, **g}, nrot)
    nblk = -(-w.T // w.chunk)
    hists = [(torch.empty((w.B, w.H, nblk, w.d, w.hidden), dtype=s["Q"].dtype, device="cuda"),
              torch.empty((w.B, w.H, nblk, w.hidden, w.d), dtype=s["Q"].dtype, device="cuda")) for s in sets]
    fwd_out = [(torch.empty_like(s["Q"]), torch.empty_like(s["W1"]), torch.empty_like(s["W2"])) for s in sets]
    bwd_out = [(torch.empty_like(s["Q"]), torch.empty_like(s["Q"]), torch.empty_like(s["Q"]),
                torch.empty_like(s["eta"]), torch.empty_like(s["W1"]), torch.empty_like(s["W2"])) for s in sets]

    def fwd(i):
        s, (Z, A, Bm), (H1, H2) = sets[i % nrot], fwd_out[i % nrot], hists[i % nrot]
        T_mod.ttt_mlp_prefill_hist(s["Q"], s["K"], s["V"], s["eta"], s["W1"], s["W2"], Z, A, Bm, H1, H2, w.chunk)

    def bwd(i):
        s, o, (H1, H2) = sets[i % nrot], bwd_out[i % nrot], hists[i % nrot]
        T_mod.ttt_mlp_prefill_backward(s["Q"], s["K"], s["V"], s["eta"], H1, H2, s["dZ"], s["dW1T"], s["dW2T"], *o,
                                       w.chunk)

    for i in range(nrot):
        fwd(i)
    ms_f, ms_f_launch = timed_loop(fwd, steps, warmup, world)
    ms_b, ms_b_launch = timed_loop(bwd, steps, warmup, world)
    # the library's choice for this shape (include/ttt.h): warp-level MMAs for bf16, d 64, hidden 256,
    # chunk 16, unless TTT_MLP_BACKWARD_KERNEL=simt
    mma = (w.dtype == "bf16" and w.d == 64 and w.hidden == 256 and w.chunk == 16 and w.T % 16 == 0
           and os.environ.get("TTT_MLP_BACKWARD_KERNEL") != "simt")
    backward_kernel = "warp-level MMA, bf16 operands" if mma else "SIMT fp32"
    nbytes = mlp_backward_bytes(w.B, w.H, w.T, w.d, w.hidden, w.chunk)
    flops = mlp_backward_flops(w.B, w.H, w.T, w.d, w.hidden, w.chunk)
    t_roof = max(nbytes / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
    del sets, hists, fwd_out, bwd_out
    return {"tokens_per_s": w.B * w.T / ((ms_f + ms_b) * 1e-3), "ms_per_step": ms_f + ms_b,
            "forward_hist_ms_per_launch": ms_f_launch, "backward_ms_per_launch": ms_b_launch,
            "backward_bytes_per_launch": nbytes, "backward_flops_per_launch": flops,
            "backward_roofline_us": t_roof * 1e6, "backward_frac": t_roof / (ms_b_launch * 1e-3),
            "backward_frac_of_rated": rated_roof(nbytes, flops) / (ms_b_launch * 1e-3),
            "bound": "hbm" if nbytes / (peaks["hbm_gbs"] * 1e9) > flops / (peaks["bf16_tflops"] * 1e12) else "tensor",
            "backward_kernel": backward_kernel}


def bench_decode(T_mod, w, steps, warmup, world, peaks, graph_steps=1024, nrot=NROT):
    """A CUDA graph of `graph_steps` decode steps; `nrot` state copies rotate so the state streams from HBM."""
    x = WL.decode_inputs(w.B, w.H, w.d, graph_steps, w.seed)
    q, k, v, e = (x[n].cuda() for n in ("q", "k", "v", "eta"))
    states = [x["W"].cuda() for _ in range(nrot)]
    z = torch.empty_like(q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # one eager pass also serves as warm-up of the library
        for i in range(2):
            T_mod.ttt_linear_decode_step(q[i], k[i], v[i], e[i], states[i % nrot], z[i])
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(graph_steps):
            T_mod.ttt_linear_decode_step(q[i], k[i], v[i], e[i], states[i % nrot], z[i])
    ms, ms_launch = timed_loop(lambda i: g.replay(), steps, warmup, world, graph=False)
    per_step = ms_launch / graph_steps
    nbytes = decode_bytes(w.B, w.H, w.d)
    state_bytes = 2 * w.B * w.H * w.d * w.d * 4
    t_roof = nbytes / (peaks["hbm_gbs"] * 1e9)
    return {"tokens_per_s": w.B / (per_step * 1e-3), "us_per_step": per_step * 1e3, "graph_steps": graph_steps,
            "bytes_per_step": nbytes, "achieved_gbs": nbytes / (per_step * 1e-3) / 1e9,
            "state_gbs": state_bytes / (per_step * 1e-3) / 1e9, "roofline_us": t_roof * 1e6,
            "frac": t_roof / (per_step * 1e-3), "bound": "hbm", "state_copies": nrot,
            "frac_of_rated": rated_roof(nbytes, 0) / (per_step * 1e-3)}


def mlp_decode_bytes(B, H, d, hd, elt=2):
    """Per step: W1 and W2 read + written once, q,k,v read, z written, eta read."""
    return 2 * 2 * B * H * d * hd * 4 + 4 * B * H * d * elt + 4 * B * H


def bench_mlp_decode(T_mod, w, steps, warmup, world, peaks, graph_steps=256, nrot=2):
    """A CUDA graph of `graph_steps` TTT-MLP decode steps; `nrot` state copies rotate (2 x 100.7 MB > L2)."""
    x = WL.mlp_decode_inputs(w.B, w.H, w.d, w.hidden, graph_steps, w.seed)
    q, k, v, e = (x[n].cuda() for n in ("q", "k", "v", "eta"))
    states = [(x["W1"].cuda(), x["W2"].cuda()) for _ in range(nrot)]
    z = torch.empty_like(q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(2):
            W1, W2 = states[i % nrot]
            T_mod.ttt_mlp_decode_step(q[i], k[i], v[i], e[i], W1, W2, z[i])
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(graph_steps):
            W1, W2 = states[i % nrot]
            T_mod.ttt_mlp_decode_step(q[i], k[i], v[i], e[i], W1, W2, z[i])
    ms, ms_launch = timed_loop(lambda i: g.replay(), steps, warmup, world, graph=False)
    per_step = ms_launch / graph_steps
    nbytes = mlp_decode_bytes(w.B, w.H, w.d, w.hidden)
    t_roof = nbytes / (peaks["hbm_gbs"] * 1e9)
    return {"tokens_per_s": w.B / (per_step * 1e-3), "us_per_step": per_step * 1e3, "graph_steps": graph_steps,
            "bytes_per_step": nbytes, "achieved_gbs": nbytes / (per_step * 1e-3) / 1e9,
            "roofline_us": t_roof * 1e6, "frac": t_roof / (per_step * 1e-3), "bound": "hbm", "state_copies": nrot,
            "frac_of_rated": rated_roof(nbytes, 0) / (per_step * 1e-3)}


def bench_e2e(T_mod, w, steps, warmup, world):
    """Public API with pinned host buffers, every step: H2D of the step's inputs, the prefill, D2H of Z and W.

    Steps are pipelined the way a serving loop would run them: three streams (upload, compute, download)
    and two device buffer sets, so that the upload of step i + 1 and the download of step i - 1 overlap
    the prefill of step i (PCIe carries both directions at once).  The timed region opens with an event
    on the upload stream, before any of its work, and closes on the current stream after it has joined
    the last download; every step's copies and its prefill fall inside it."""
    x = WL.workload_inputs(w)
    host = {k: v.pin_memory() for k, v in x.items()}
    dev = [{k: torch.empty_like(v, device="cuda") for k, v in x.items()} for _ in range(2)]
    outs = [(torch.empty_like(dev[0]["Q"]), torch.empty_like(dev[0]["W0"])) for _ in range(2)]
    Zh = torch.empty_like(host["Q"]).pin_memory()
    Wh = torch.empty_like(host["W0"]).pin_memory()
    ws = T_mod.linear_workspace(dev[0]["Q"], w.chunk)  # scratch, allocated once like any workspace
    s_up, s_cmp, s_dn = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    # set b: uploaded, computed, downloaded (each records once per use of the set)
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_dn = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        b = i % 2
        d, (Z, W) = dev[b], outs[b]
        s_up.wait_event(ev_cmp[b])  # the prefill of step i - 2 has read set b
        with torch.cuda.stream(s_up):
            for k in d:
                d[k].copy_(host[k], non_blocking=True)
        ev_up[b].record(s_up)
        s_cmp.wait_event(ev_up[b])
        s_cmp.wait_event(ev_dn[b])  # the download of step i - 2 has read Z, W of set b
        T_mod.ttt_linear_prefill_ws(d["Q"], d["K"], d["V"], d["eta"], d["W0"], Z, W, w.chunk, ws, stream=s_cmp)
        ev_cmp[b].record(s_cmp)
        s_dn.wait_event(ev_cmp[b])
        with torch.cuda.stream(s_dn):
            Zh.copy_(Z, non_blocking=True)
            Wh.copy_(W, non_blocking=True)
        ev_dn[b].record(s_dn)

    for i in range(max(warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    t0.record(s_up)
    for i in range(steps):
        step(i)
    for st in (s_up, s_cmp, s_dn):
        cur.wait_stream(st)
    t1.record(cur)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(t0.elapsed_time(t1) / steps, world)
    # the pipelined steps deliver what one plain call on the same inputs gives, bit for bit
    Zr, Wr = torch.empty_like(outs[0][0]), torch.empty_like(outs[0][1])
    T_mod.ttt_linear_prefill_ws(dev[0]["Q"], dev[0]["K"], dev[0]["V"], dev[0]["eta"], dev[0]["W0"], Zr, Wr,
                                w.chunk, ws)
    torch.cuda.synchronize()
    if not (torch.equal(Zr.cpu(), Zh) and torch.equal(Wr.cpu(), Wh)):
        raise RuntimeError("pipelined end-to-end steps disagree with a plain call")
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = Zh.numel() * Zh.element_size() + Wh.numel() * Wh.element_size()
    # what the host link gives for the same bytes in the same run: the step's uploads alone, and its
    # uploads and downloads at once (the lower bound of a pipelined step)
    def copies(down):
        with torch.cuda.stream(s_up):
            for k in dev[0]:
                dev[0][k].copy_(host[k], non_blocking=True)
        if down:
            with torch.cuda.stream(s_dn):
                Zh.copy_(outs[0][0], non_blocking=True)
                Wh.copy_(outs[0][1], non_blocking=True)
    link = {}
    for name, down in (("h2d_ms", False), ("h2d_with_d2h_ms", True)):
        copies(down)
        torch.cuda.synchronize()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_up)
        s_dn.wait_event(a)
        for _ in range(20):
            copies(down)
        for st in (s_up, s_dn):
            cur.wait_stream(st)
        z.record(cur)
        torch.cuda.synchronize()
        link[name] = a.elapsed_time(z) / 20
    link["h2d_gbs"] = h2d / (link["h2d_ms"] * 1e6)
    return {"value": w.B * w.T / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "pipelining": "upload, prefill and download on three streams, two device buffer sets",
            "host_link": link}


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


def oracle_single_thread(O, flat, chunk, T, H):
    """tokens/s of the oracle's dual form on one (batch, head) sequence with one thread (restores the
    count); a token carries H heads, so one sequence of T tokens is T / H tokens of the workload."""
    n0 = O.num_threads()
    O.set_num_threads(1)
    try:
        one = {k: v[:, :1] for k, v in flat.items()}
        t0 = time.perf_counter()
        O.linear_dual(one["Q"], one["K"], one["V"], one["eta"], one["W0"], chunk)
        dt = time.perf_counter() - t0
    finally:
        O.set_num_threads(n0)
    return {"value": T / H / dt, "unit": "tokens/s", "cores": 1, "seconds": dt,
            "sample": f"fp64 dual form on 1 (batch, head) sequence ({T} tokens, one of {H} heads), 1 thread"}


def oracle_flat(w):
    x = WL.workload_inputs(w)
    r = {k: WL.to_f64(v) for k, v in x.items()}
    BH = w.B * w.H
    return {k: v.reshape((1, BH) + v.shape[2:]) for k, v in r.items()}


def cpu_baseline(w, target_s=12.0, heads=None):
    """The fp64 oracle (dual form) on a sample of the workload's heads (all of them when they fit in
    about target_s seconds), plus the same oracle on one thread and the CPU model."""
    from oracle import oracle as O
    flat = oracle_flat(w)
    BH = w.B * w.H
    n = heads or 1
    while True:
        sub = {k: v[:, :n] for k, v in flat.items()}
        t0 = time.perf_counter()
        O.linear_dual(sub["Q"], sub["K"], sub["V"], sub["eta"], sub["W0"], w.chunk)
        dt = time.perf_counter() - t0
        if heads or dt * 2 >= target_s or n >= BH:
            break
        n = min(BH, max(n + 1, int(n * min(8.0, target_s / max(dt, 1e-3)))))
    return {"value": n * w.T / w.H / dt, "unit": "tokens/s", "cores": O.num_threads(), "kind": "oracle",
            "sample": f"fp64 dual form on {n} of {BH} (batch, head) sequences of the {w.name} workload "
                      f"({w.T} tokens each, {dt:.2f} s)", "seconds": dt, "cpu_model": cpu_model(),
            "single_thread": oracle_single_thread(O, flat, w.chunk, w.T, w.H)}


def run_ours(args):
    rank, world = dist_setup(args.gpus)
    from test_sequence_layers_07_b300 import ttt as T_mod
    T_mod.load_library()
    peaks, peaks_kind = load_peaks()
    w = WL.WORKLOADS["linear_prefill"]
    dev = torch.cuda.current_device()
    sampler = ClockSampler(dev)
    head = bench_linear(T_mod, w, w.chunk, args.steps, args.warmup, world, peaks, sampler=sampler)
    clocks = sampler.summary()
    value = world * w.B * w.T / (head["ms_per_step"] * 1e-3)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "TTT-Linear prefill B=8 H=12 d=64 T=2048 chunk=16 (bf16 Q/K/V/Z, fp32 state)",
                   "path": head["path"],
                   "global_batch": w.B * world, "seq_len": w.T, "heads": w.H, "head_dim": w.d, "chunk": w.chunk,
                   "parallelism": f"dp{world}" if world > 1 else "single-gpu",
                   "l2": f"{NROT} rotating input copies ({NROT * linear_bytes(w.B, w.H, w.T, w.d) / 1e6:.0f} MB > "
                         f"126 MB L2)",
                   "timing": "the K steps replayed as one CUDA graph, CUDA events around the replay" if GRAPH
                             else "per-call launches, CUDA events around the K steps"},
        "roofline": {"bound": "hbm", "achieved": head["achieved_gbs"],
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": head["achieved_gbs"] / peaks["hbm_gbs"],
                     "traffic": ncu_traffic("linear_prefill", LINEAR_SRC),
                     "peak_kind": f"{peaks_kind} copy bandwidth",
                     "frac_of_rated": head["achieved_gbs"] / RATED_PEAKS["hbm_gbs"],
                     "rated_peak": RATED_PEAKS["hbm_gbs"], "bytes_per_launch": head["bytes_per_launch"],
                     "ms_per_launch": head["ms_per_launch"]},
        "clocks": clocks,
        "gpu_launches": args.steps * head["kernel_launches_per_call"],
    }
    if not args.no_e2e:
        line["e2e"] = bench_e2e(T_mod, w, max(5, min(200, args.steps // 10)), args.warmup, world)
    if args.rows != "none":
        want = lambda name: args.rows in ("all", name)
        rows = {"linear_prefill": head}
        rsteps = max(5, min(50, args.steps // 20))
        if want("linear_split"):
            # few heads, long sequence: where the one-pass scan leaves most SMs idle and the split
            # along the sequence pays; both paths timed on the same inputs
            wf = WL.WORKLOADS["linear_few_heads"]
            rows["linear_few_heads_one_pass"] = bench_linear(T_mod, wf, wf.chunk, rsteps, args.warmup, world, peaks,
                                                             nrot=2)
            rows["linear_few_heads_split"] = bench_linear(T_mod, wf, wf.chunk, rsteps, args.warmup, world, peaks,
                                                          nrot=2, split=True)
        if want("mlp_prefill"):
            rows["mlp_prefill"] = bench_mlp(T_mod, WL.WORKLOADS["mlp_prefill"], rsteps, args.warmup, world, peaks)
        if want("long_context"):
            wl = WL.WORKLOADS["long_context"]
            for b in wl.chunks:
                rows[f"long_context_b{b}"] = bench_linear(T_mod, wl, b, rsteps, args.warmup, world, peaks, nrot=1)
        if want("decode"):
            wd = WL.WORKLOADS["decode"]
            rows["decode"] = bench_decode(T_mod, wd, max(3, rsteps // 5), args.warmup, world, peaks)
        if want("mlp_decode"):
            wd = WL.WORKLOADS["mlp_decode"]
            rows["mlp_decode"] = bench_mlp_decode(T_mod, wd, max(3, rsteps // 5), args.warmup, world, peaks)
        if want("mlp_backward"):
            rows["mlp_backward"] = bench_mlp_backward(T_mod, WL.WORKLOADS["mlp_prefill"], 3, args.warmup, world,
                                                      peaks)
        if want("momentum"):
            rows["linear_momentum"] = bench_momentum(T_mod, w, 0.9, max(3, rsteps // 5), args.warmup, world, peaks)
        if want("backward"):
            rows["linear_backward"] = bench_backward(T_mod, w, max(3, rsteps // 5), args.warmup, world, peaks)
        line["rows"] = rows
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args, budget_s=150.0):
    """The fp64 oracle's dual form on the host cores, timed per step.  A step is the whole headline
    workload (all B*H sequences) when warm-up + steps fit in about budget_s seconds, else the largest
    whole multiple of the thread count of its sequences that does (every core busy); the line
    reports the measured time of those steps and the tokens they processed, not an extrapolation."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import oracle as O
    w = WL.WORKLOADS["linear_prefill"]
    flat = oracle_flat(w)
    BH = w.B * w.H
    cores = O.num_threads()
    t0 = time.perf_counter()  # calibration: one untimed pass over every sequence
    O.linear_dual(flat["Q"], flat["K"], flat["V"], flat["eta"], flat["W0"], w.chunk)
    per_seq = (time.perf_counter() - t0) / BH
    n = BH
    if (args.warmup + args.steps) * per_seq * BH > budget_s:
        n = int(budget_s / ((args.warmup + args.steps) * per_seq))
        n = min(BH, max(min(cores, BH), n // cores * cores))
    sub = {k: v[:, :n] for k, v in flat.items()}
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        O.linear_dual(sub["Q"], sub["K"], sub["V"], sub["eta"], sub["W0"], w.chunk)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    step_s = sum(times) / len(times)
    value = n * w.T / w.H / step_s  # a token carries H heads: n sequences are n T / H tokens
    sample = (f"fp64 oracle dual form on {n} of the {BH} (batch, head) sequences of the workload per step "
              f"({n * w.T / w.H:g} tokens), {cores} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "TTT-Linear prefill B=8 H=12 d=64 T=2048 chunk=16", "global_batch": w.B,
                       "seq_len": w.T, "sequences_per_step": n, "tokens_per_step": n * w.T / w.H},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model(),
                             "single_thread": oracle_single_thread(O, flat, w.chunk, w.T, w.H)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# sources of the headline kernel (the one-pass d = 64 prefill): the committed DRAM traffic counts only while
# they are unchanged
LINEAR_SRC = ["linear_prefill_fused.cu", "ptx.cuh", "ttt_common.cuh"]


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--eager", action="store_true",
                    help="time per-call launches instead of replaying the timed steps as a CUDA graph")
    ap.add_argument("--rows", choices=["all", "none", "linear_split", "mlp_prefill", "long_context",
                                       "decode", "mlp_decode", "backward", "momentum", "mlp_backward"],
                    default="all",
                    help="workload rows timed after the headline (default: all)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args(argv)
    global GRAPH
    GRAPH = not args.eager
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    args.steps = max(1, args.steps)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
