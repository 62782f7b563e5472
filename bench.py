"""Benchmark of the DeepSeekMoE layer forward on B300.

One step = one pass of the whole layer (router logits, route, dispatch,
expert FFNs, combine) over one batch of T seeded synthetic tokens whose
inputs are already resident in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the same workload

The headline workload is the DeepSeek-V3-shaped prefill layer (the largest
layer that fits one GPU); the same run also times the decode-shaped layer and
the DeepSeekMoE-16B-shaped layer (with its backward) and reports them under
"workloads", each with its own roofline and clock record.

Under torchrun every rank runs an independent replica of the layer on its own
GPU (tokens are independent, so the layer shards by batch with no exchange);
value = all tokens processed / the slowest rank's time.  ``--gpus N`` without
torchrun relaunches the script under torchrun with N processes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fine_grained_shared_gemm_b300 import moe as M          # noqa: E402
from fine_grained_shared_gemm_b300 import workloads as W    # noqa: E402

DEFAULT_WORKLOAD = "v3_prefill_bf16"
# timed in the same run as the headline, after it
EXTRA_WORKLOADS = ("decode_bf16", "dsmoe16b_bf16")
# the backward is timed on this layer (the V3-shaped backward needs ~80 GB of
# gradients and scratch besides the weights)
BACKWARD_WORKLOAD = "dsmoe16b_bf16"
METRIC = "MoE layer tokens/s & TFLOP/s (% bf16 peak); decode weight GB/s (% HBM)"
L2_FLUSH_BYTES = 512 << 20     # larger than the 126 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# nominal dense bf16 rate and HBM bandwidth of one B300, as the workload's
# targets are stated against (reported beside the measured-peak fractions)
NOMINAL = {"bf16_tflops": 2250.0, "hbm_gbs": 8000.0}
PEAK_NOTE = ("hbm_gbs is a device copy rate counting read + write bytes; a kernel that "
             "mostly reads can exceed it")


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over all ranks (the slowest rank's time)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_rank: int, seconds: float, world: int, device):
    """(tokens/s over all ranks, slowest rank's seconds): every rank processed
    tokens_per_rank tokens; the job took as long as its slowest rank."""
    slowest = max_over_ranks(seconds, device)
    return tokens_per_rank * world / slowest, slowest


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


def expert_flops(s: W.MoEShape) -> int:
    return s.T * (s.top_k + s.n_shared) * s.n_mats * 2 * s.H * s.inter


def used_experts(s: W.MoEShape, offsets: np.ndarray) -> int:
    """Experts whose weights a step reads: routed experts with a token, and
    every shared expert."""
    return int((np.diff(offsets) > 0).sum()) + s.n_shared


def touched_weight_bytes(s: W.MoEShape, offsets: np.ndarray) -> int:
    """Expert weights a step must read at least once: every expert with a token."""
    return used_experts(s, offsets) * s.n_mats * s.H * s.inter * 2


def ffn_alg_bytes(s: W.MoEShape, offsets: np.ndarray) -> int:
    """Bytes one moe_expert_ffn call must move at least: every expert with a
    token reads its weights once; the expert input rows come in (the permuted
    rows, and u once per shared expert), the activation goes out and back
    in, the outputs go out."""
    e = 2 if s.dtype == "bf16" else 4
    rows = s.T * (s.top_k + s.n_shared)
    return (used_experts(s, offsets) * s.n_mats * s.H * s.inter + rows * s.H * 2
            + rows * s.inter * 2) * e


def decode_alg_bytes(s: W.MoEShape, offsets: np.ndarray) -> int:
    """Bytes one decode-shaped layer step must move at least: the weights of
    every expert with a token, the routing centroids, the tokens in and the
    output out."""
    e = 2 if s.dtype == "bf16" else 4
    return touched_weight_bytes(s, offsets) * e // 2 + s.n_routed * s.H * e + 2 * s.T * s.H * e


def is_decode(s: W.MoEShape) -> bool:
    """Decode-shaped: fewer routed rows than two per expert, so the step is
    bound by streaming the touched experts' weights from HBM."""
    return s.T * s.top_k < 2 * s.n_routed


def prefill_roofline(s: W.MoEShape, offsets: np.ndarray, ffn_s: float, peaks: dict) -> dict:
    """The expert FFN (both grouped GEMMs, one moe_expert_ffn call of ffn_s
    seconds) against the measured dense bf16 tensor peak (burst: the call is
    timed on its own and lasts milliseconds), with the HBM roof of its
    algorithmic bytes under other_roof."""
    flops = expert_flops(s)
    alg_bytes = ffn_alg_bytes(s, offsets)
    tf = flops / ffn_s / 1e12
    gb = alg_bytes / ffn_s / 1e9
    t_flops = flops / (peaks["bf16_tflops"] * 1e12)
    t_bytes = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    r = {"bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_tflops"],
         "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
         "frac_of_nominal": round(tf / NOMINAL["bf16_tflops"], 4),
         "algorithmic_flop": flops}
    if peaks.get("bf16_tflops_sustained"):
        # the same against the rate measured under a seconds-long load at the
        # power cap, for a call that ran power-capped (see the clocks record)
        r["peak_sustained"] = peaks["bf16_tflops_sustained"]
        r["frac_of_sustained"] = round(tf / peaks["bf16_tflops_sustained"], 4)
    r.update({
            "other_roof": {"bound": "hbm", "achieved": round(gb, 1), "peak": peaks["hbm_gbs"],
                           "unit": "GB/s", "frac": round(gb / peaks["hbm_gbs"], 4),
                           "algorithmic_bytes": alg_bytes},
            "ridge": "memory side" if t_bytes > t_flops else "tensor side"})
    return r


def decode_roofline(s: W.MoEShape, offsets: np.ndarray, layer_s: float, ffn_s: float,
                    peaks: dict) -> dict:
    """A decode-shaped layer against HBM: its algorithmic bytes over the whole
    layer's time (one step), with the expert FFN's weight stream over the FFN
    call's time alongside."""
    b = decode_alg_bytes(s, offsets)
    gb = b / layer_s / 1e9
    w = touched_weight_bytes(s, offsets)
    gb_ffn = w / ffn_s / 1e9
    r = {"bound": "hbm", "achieved": round(gb, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
         "frac": round(gb / peaks["hbm_gbs"], 4),
         "frac_of_nominal": round(gb / NOMINAL["hbm_gbs"], 4), "algorithmic_bytes": b,
         "experts_touched": used_experts(s, offsets),
         "ffn_only": {"achieved": round(gb_ffn, 1), "unit": "GB/s",
                      "frac": round(gb_ffn / peaks["hbm_gbs"], 4), "weight_bytes": w}}
    if gb > peaks["hbm_gbs"] or gb_ffn > peaks["hbm_gbs"]:
        r["note"] = PEAK_NOTE
    return r


def kernel_source_hash() -> str:
    src = os.path.join(ROOT, "fine_grained_shared_gemm_b300", "csrc", "tc_gemm.cuh")
    with open(src, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per expert-FFN call from the committed ncu summary, if it was
    taken on the current tensor-core kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "expert_ffn_dram_traffic.txt")
    if not os.path.exists(p):
        return None
    want = kernel_source_hash()
    for line in open(p):
        parts = line.split()
        if len(parts) >= 3 and parts[0] == workload and parts[1] == want:
            return float(parts[2])
    return None


class _Nvml:
    """Read-only NVML queries through ctypes (libnvidia-ml ships with the
    driver; the pynvml wrapper may be absent)."""

    CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        self._check(self.lib.nvmlInit_v2(), "nvmlInit_v2")

    def _check(self, rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} returned {rc}")

    def handle_for_uuid(self, uuid: str):
        c = self.c
        n = c.c_uint(0)
        self._check(self.lib.nvmlDeviceGetCount_v2(c.byref(n)), "nvmlDeviceGetCount_v2")
        handles = []
        for i in range(n.value):
            h = c.c_void_p()
            self._check(self.lib.nvmlDeviceGetHandleByIndex_v2(c.c_uint(i), c.byref(h)),
                        "nvmlDeviceGetHandleByIndex_v2")
            buf = c.create_string_buffer(96)
            self._check(self.lib.nvmlDeviceGetUUID(h, buf, c.c_uint(96)), "nvmlDeviceGetUUID")
            if uuid in buf.value.decode():
                return h
            handles.append(h)
        if len(handles) == 1:
            return handles[0]
        raise RuntimeError(f"no NVML device with uuid {uuid}")

    def sm_clock(self, h) -> int:
        v = self.c.c_uint(0)
        self._check(self.lib.nvmlDeviceGetClockInfo(h, self.CLOCK_SM, self.c.byref(v)),
                    "nvmlDeviceGetClockInfo")
        return v.value

    def sm_max_clock(self, h) -> int:
        v = self.c.c_uint(0)
        self._check(self.lib.nvmlDeviceGetMaxClockInfo(h, self.CLOCK_SM, self.c.byref(v)),
                    "nvmlDeviceGetMaxClockInfo")
        return v.value

    def event_reasons(self, h) -> int:
        v = self.c.c_ulonglong(0)
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self._check(fn(h, self.c.byref(v)), "nvmlDeviceGetCurrentClocksEventReasons")
        return v.value


class L2Flush:
    """Empties L2 between timed launches: writes a buffer larger than L2,
    then reads a second one, so that the written lines go back to HBM before
    the timed launch starts instead of during it.  The timed launch finds an
    L2 that holds none of its data and nothing dirty."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


class ClockSampler:
    """SM clock and throttle reasons sampled through NVML every 2 ms while the
    timed region runs (read-only queries; no setting is changed)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device: torch.device):
        self.device = device
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self._stop = None
        self.error = None

    def __enter__(self):
        import threading
        try:
            nv = _Nvml()
            h = nv.handle_for_uuid(str(torch.cuda.get_device_properties(self.device).uuid))
            self.max_mhz = nv.sm_max_clock(h)
        except Exception as e:   # no NVML: report the clocks as unsampled
            self.error = f"{type(e).__name__}: {e}"
            return self
        self._stop = threading.Event()

        def loop():
            while not self._stop.is_set():
                try:
                    self.samples.append(nv.sm_clock(h))
                    bits = nv.event_reasons(h)
                    for b, name in self.REASONS.items():
                        if bits & b:
                            self.reasons.add(name)
                except Exception as e:
                    self.error = f"{type(e).__name__}: {e}"
                self._stop.wait(0.002)
        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()
        return self

    def __exit__(self, *a):
        if self._stop is not None:
            self._stop.set()
            self._thread.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"],
                    "error": self.error}
        return {"sm_mhz": statistics.median(self.samples),
                "sm_mhz_mean": round(statistics.fmean(self.samples), 1),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples)}


class Layer:
    """Device buffers and the five C-ABI calls of one layer step."""

    def __init__(self, shape: W.MoEShape, dev):
        self.s = s = shape
        self.inp = W.make_inputs(shape, dev, seed=0)
        self.wt = M.weights_struct(self.inp)
        T, E, k, Ks, H = s.T, s.n_routed, s.top_k, s.n_shared, s.H
        dt = s.torch_dtype
        self.logits = torch.empty((T, E), dtype=torch.float32, device=dev)
        self.idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.w = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.off = torch.empty((E + 1,), dtype=torch.int32, device=dev)
        self.row_token = torch.empty((T * k,), dtype=torch.int32, device=dev)
        self.slot_row = torch.empty((T * k,), dtype=torch.int32, device=dev)
        self.u_perm = torch.empty((T * k, H), dtype=dt, device=dev)
        self.y_perm = torch.empty((T * k, H), dtype=dt, device=dev)
        self.y_shared = torch.empty((Ks, T, H), dtype=dt, device=dev)
        self.h = torch.empty((T, H), dtype=dt, device=dev)
        self.ws_d = M.alloc_workspace(M.moe_dispatch_workspace_size(s), dev)
        self.ws_f = M.alloc_workspace(M.moe_expert_ffn_workspace_size(s), dev)
        self.ws_l = M.alloc_workspace(M.moe_layer_workspace_size(s), dev)
        self.ws_r = M.alloc_workspace(M.moe_router_logits_workspace_size(s), dev)
        self.launches_per_step = forward_launches(s)

    def step(self, ev=None):
        s, i = self.s, self.inp
        M.moe_router_logits(s, i.u, i.centroids, i.logit_offset, self.logits, self.ws_r)
        M.moe_route(s, self.logits, i.select_bias, self.idx, self.w)
        M.moe_dispatch(s, self.idx, i.u, self.off, self.row_token, self.slot_row, self.u_perm,
                       self.ws_d)
        if ev is not None:
            ev[0].record()
        M.moe_expert_ffn(s, self.wt, i.u, self.u_perm, self.off, self.y_perm, self.y_shared,
                         self.ws_f)
        if ev is not None:
            ev[1].record()
        M.moe_combine(s, i.u, self.y_perm, self.y_shared, self.w, self.slot_row, self.h)


def sustained_frac(flops: float, ms: float, peaks: dict):
    """flops in ms against the bf16 rate measured under a seconds-long load
    at the power cap (None without that figure)."""
    p = peaks.get("bf16_tflops_sustained")
    return round(flops / (ms / 1e3) / 1e12 / p, 4) if p else None


def backward_launches(s: W.MoEShape, saved: bool = False) -> int:
    """Kernel launches of one moe_layer_backward call (counted from its host
    code); saved: the call reuses moe_layer_forward_train's tensors."""
    sw = s.act == W.ACT_SWIGLU
    k = s.top_k > 0
    rows = k or s.n_shared > 0                    # any expert input rows at all
    n = 0
    if not saved:
        n += 2 + (4 if k else 1)                  # router logits, route, dispatch
        n += (2 if sw else 1) if rows else 0      # pre-activations recomputed
    n += 2 if k else 0                            # scatter dh rows, row gate weights
    n += 2                                        # FFN plan, weight-gradient plan
    n += 1 if rows else 0                         # dm = dh W2 (SwiGLU: + derivative)
    if not sw:
        n += s.n_shared + (1 if k else 0)         # ReLU derivative
    n += 1 + 2 + 1                                # gate, router GEMMs, partial sums
    n += (1 if rows else 0) + 1                   # dx, du
    n += 2                                        # weight-gradient GEMMs
    return n


def router_splits(s: W.MoEShape) -> int:
    """Contraction ranges of the layer's router-logits GEMM (the library's
    rule: bf16 batches with few 128-expert x 64-token tiles cut H so that
    about 128 CTAs stream it, in whole two-k-block stages, at most 32)."""
    if s.dtype != "bf16" or s.T <= 0:
        return 1
    cdiv = lambda a, b: -(-a // b)
    tiles = cdiv(s.n_routed, 128) * cdiv(s.T, 64)
    nkb = cdiv(s.H, 64)
    want = min(32, 128 // tiles, nkb // 2)
    if want < 2:
        return 1
    per = 2 * cdiv(nkb, want * 2)
    n = cdiv(nkb, per)
    return n if n >= 2 else 1


def forward_launches(s: W.MoEShape) -> int:
    """Kernel launches of one moe_layer_forward(_train) call (one more, the
    partial logits' sum, when the router GEMM is split)."""
    return (10 if s.top_k > 0 else 7) + (1 if router_splits(s) > 1 else 0)


def measure_backward(args, shape, layer, flush, dev, peaks):
    """moe_layer_backward at the same workload: device time per call (L2
    flushed between calls), algorithmic FLOPs = 2 x the forward's expert
    FLOPs (input and weight gradients) + 4·T·E·H for the router."""
    need = M.moe_layer_backward_workspace_size(shape)
    if need == 0:
        return None
    s, inp = shape, layer.inp
    E, Ks, H, I = s.n_routed, s.n_shared, s.H, s.inter
    sw = s.act == W.ACT_SWIGLU
    f = lambda *d: torch.empty(d, dtype=torch.float32, device=dev)
    g = [f(E, H), f(E, I, H), f(E, I, H) if sw else None, f(E, H, I),
         f(Ks, I, H) if Ks else None, f(Ks, I, H) if Ks and sw else None,
         f(Ks, H, I) if Ks else None]
    grads = M.weight_grads(*g)
    ws = M.alloc_workspace(need, dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1)
    dh = torch.randn((s.T, H), generator=gen, device=dev).to(s.torch_dtype)
    du = torch.empty_like(dh)
    for _ in range(args.warmup):
        M.moe_layer_backward(s, layer.wt, inp.u, dh, du, grads, ws)
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    with ClockSampler(dev) as clk_b:
        for i in range(K):
            flush()
            ev[i][0].record()
            M.moe_layer_backward(s, layer.wt, inp.u, dh, du, grads, ws)
            ev[i][1].record()
        torch.cuda.synchronize()
    st, code = M.moe_device_status()
    if st != M.MOE_OK:
        raise RuntimeError(f"device status {st} code {code} in the backward")
    ms = sum(a.elapsed_time(b) for a, b in ev) / K
    flops = 2 * expert_flops(s) + 4 * s.T * E * H
    tf = flops / (ms / 1e3) / 1e12
    # training step: the forward that keeps routing and pre-activations, then
    # the backward that reuses them (each call timed on its own, L2 flushed)
    saved = M.alloc_workspace(M.moe_layer_saved_size(s), dev)
    h = torch.empty_like(dh)
    for _ in range(args.warmup):
        M.moe_layer_forward_train(s, layer.wt, inp.u, h, saved, layer.ws_l)
        M.moe_layer_backward(s, layer.wt, inp.u, dh, du, grads, ws, saved=saved)
    torch.cuda.synchronize()
    ev_f = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(K)]
    ev_b = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(K)]
    with ClockSampler(dev) as clk_t:
        for i in range(K):
            flush()
            ev_f[i][0].record()
            M.moe_layer_forward_train(s, layer.wt, inp.u, h, saved, layer.ws_l)
            ev_f[i][1].record()
            flush()
            ev_b[i][0].record()
            M.moe_layer_backward(s, layer.wt, inp.u, dh, du, grads, ws, saved=saved)
            ev_b[i][1].record()
        torch.cuda.synchronize()
    st, code = M.moe_device_status()
    if st != M.MOE_OK:
        raise RuntimeError(f"device status {st} code {code} in the training step")
    f_ms = sum(a.elapsed_time(b) for a, b in ev_f) / K
    b_ms = sum(a.elapsed_time(b) for a, b in ev_b) / K
    step_flops = expert_flops(s) + 2 * s.T * E * H + flops
    # the same two calls captured once into CUDA graphs and replayed, as a
    # training loop over fixed shapes runs them (the same kernels; the graph
    # saves the per-launch host and launch-processing time)
    g_f, g_b = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g_f):
        M.moe_layer_forward_train(s, layer.wt, inp.u, h, saved, layer.ws_l)
    with torch.cuda.graph(g_b):
        M.moe_layer_backward(s, layer.wt, inp.u, dh, du, grads, ws, saved=saved)
    for _ in range(args.warmup):
        g_f.replay()
        g_b.replay()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk_g:
        for i in range(K):
            flush()
            ev_f[i][0].record()
            g_f.replay()
            ev_f[i][1].record()
            flush()
            ev_b[i][0].record()
            g_b.replay()
            ev_b[i][1].record()
        torch.cuda.synchronize()
    st, code = M.moe_device_status()
    if st != M.MOE_OK:
        raise RuntimeError(f"device status {st} code {code} in the graph-replayed training step")
    gf_ms = sum(a.elapsed_time(b) for a, b in ev_f) / K
    gb_ms = sum(a.elapsed_time(b) for a, b in ev_b) / K
    del g_f, g_b
    del ws, g, grads, saved
    return {"tokens_per_s": round(s.T / (ms / 1e3), 1), "ms_per_step": round(ms, 4),
            "algorithmic_tflop": round(flops / 1e12, 4), "tflops": round(tf, 1),
            "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
            "frac_of_sustained_bf16": (round(tf / peaks["bf16_tflops_sustained"], 4)
                                       if peaks.get("bf16_tflops_sustained") else None),
            "gpu_launches": backward_launches(s) * K,
            "note": "recomputes routing and the gate/up pre-activations from u; "
                    "weight gradients fp32",
            "clocks": clk_b.summary(),
            "backward_saved": {
                "ms": round(b_ms, 4),
                "tflops": round(flops / (b_ms / 1e3) / 1e12, 1),
                "frac_of_bf16_peak": round(flops / (b_ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
                "note": "the same gradients from moe_layer_forward_train's saved tensors "
                        "(timed within the training step below)"},
            "training_step": {
                "forward_train_ms": round(f_ms, 4), "backward_saved_ms": round(b_ms, 4),
                "gpu_launches": (forward_launches(s) + backward_launches(s, saved=True)) * K,
                "tokens_per_s": round(s.T / ((f_ms + b_ms) / 1e3), 1),
                "tflops": round(step_flops / ((f_ms + b_ms) / 1e3) / 1e12, 1),
                "frac_of_sustained_bf16": sustained_frac(step_flops, f_ms + b_ms, peaks),
                "clocks": clk_t.summary(),
                "note": "moe_layer_forward_train + moe_layer_backward on its saved tensors"},
            "training_step_graph": {
                "forward_train_ms": round(gf_ms, 4), "backward_saved_ms": round(gb_ms, 4),
                "gpu_launches": (forward_launches(s) + backward_launches(s, saved=True)) * K,
                "tokens_per_s": round(s.T / ((gf_ms + gb_ms) / 1e3), 1),
                "tflops": round(step_flops / ((gf_ms + gb_ms) / 1e3) / 1e12, 1),
                "frac_of_sustained_bf16": sustained_frac(step_flops, gf_ms + gb_ms, peaks),
                "clocks": clk_g.summary(),
                "note": "the same two calls, each captured into a CUDA graph and replayed"}}


def measure_forward(args, shape, dev, flush, world, peaks, barrier):
    """Time the layer forward of one workload: K steps on device-resident
    inputs (L2 flushed before each), then K steps end to end through the
    host-buffer entry point.  Returns (entry, layer)."""
    layer = Layer(shape, dev)
    for _ in range(args.warmup):
        layer.step()
    st, code = M.moe_device_status()
    if st != M.MOE_OK:
        raise RuntimeError(f"device status {st} code {code} after warm-up ({shape.name})")
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ffn_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
    barrier()
    with ClockSampler(dev) as clk:
        for i in range(K):
            flush()                       # L2 flushed between timed steps
            starts[i].record()
            layer.step(ffn_ev[i])
            ends[i].record()
        barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ffn_ms = [a.elapsed_time(b) for a, b in ffn_ev]
    value, total_s = whole_job_rate(shape.T * K, sum(step_ms) / 1e3, world, dev)

    # end to end from pinned host buffers: every step copies its tokens in and
    # its output back inside the timed region.  The K steps go through
    # moe_layer_forward_host_stream, which overlaps step b's layer with step
    # b + 1's copy in and step b - 1's copy back; one moe_layer_forward_host
    # call per step (copies and layer of a step in sequence, or in token
    # chunks for large batches) is reported beside it.
    u_host = layer.inp.u.cpu().pin_memory()
    h_host = torch.empty_like(u_host).pin_memory()
    u_dev = torch.empty_like(layer.inp.u)
    u_slots = torch.empty((2,) + tuple(layer.inp.u.shape), dtype=layer.inp.u.dtype, device=dev)
    h_slots = torch.empty_like(u_slots)
    W_ = max(1, args.warmup)
    M.moe_layer_forward_host_stream(shape, layer.wt, [u_host] * W_, [h_host] * W_, u_slots,
                                    h_slots, layer.ws_l)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    M.moe_layer_forward_host_stream(shape, layer.wt, [u_host] * K, [h_host] * K, u_slots,
                                    h_slots, layer.ws_l)
    e1.record()
    barrier()
    e2e_value, _ = whole_job_rate(shape.T * K, e0.elapsed_time(e1) / 1e3, world, dev)
    for _ in range(W_):
        M.moe_layer_forward_host(shape, layer.wt, u_host, h_host, u_dev, layer.h, layer.ws_l)
    barrier()
    e0.record()
    for _ in range(K):
        M.moe_layer_forward_host(shape, layer.wt, u_host, h_host, u_dev, layer.h, layer.ws_l)
    e1.record()
    barrier()
    e2e_call_value, _ = whole_job_rate(shape.T * K, e0.elapsed_time(e1) / 1e3, world, dev)
    st, code = M.moe_device_status()
    if st != M.MOE_OK:
        raise RuntimeError(f"device status {st} code {code} ({shape.name})")

    ffn_s = sum(ffn_ms) / len(ffn_ms) / 1e3
    layer_s = sum(step_ms) / len(step_ms) / 1e3
    offsets = layer.off.cpu().numpy()
    flops = expert_flops(shape)
    graph_entry = None
    if is_decode(shape):
        roof = decode_roofline(shape, offsets, layer_s, ffn_s, peaks)
        roof["kernel"] = f"moe_layer_forward (all {layer.launches_per_step} launches of one step)"
    else:
        roof = prefill_roofline(shape, offsets, ffn_s, peaks)
        roof["kernel"] = "moe_expert_ffn (gate/up and down grouped GEMMs)"
    roof.update({"traffic": recorded_traffic(shape.name),
                 "peak_source": f"{peaks.get('_source', 'measured')} (burst)",
                 "ms_per_launch": round((layer_s if is_decode(shape) else ffn_s) * 1e3, 4)})
    if is_decode(shape):
        # the same step captured once into a CUDA graph and replayed, as a
        # decode loop over fixed shapes runs it (the same kernels)
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            layer.step()
        for _ in range(max(1, args.warmup)):
            g.replay()
        barrier()
        for i in range(K):
            flush()
            starts[i].record()
            g.replay()
            ends[i].record()
        barrier()
        st, code = M.moe_device_status()
        if st != M.MOE_OK:
            raise RuntimeError(f"device status {st} code {code} in the graph replays")
        g_s = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / K / 1e3
        g_roof = decode_roofline(shape, offsets, g_s, ffn_s, peaks)
        graph_entry = {"ms_per_step": round(g_s * 1e3, 4),
                       "tokens_per_s": round(shape.T / g_s, 1),
                       "achieved": g_roof["achieved"], "unit": g_roof["unit"],
                       "frac": g_roof["frac"],
                       "note": "the layer step captured into a CUDA graph and replayed"}
        del g
    entry = {
        "value": round(value, 1), "unit": "tokens/s",
        "ms_per_step": round(total_s / K * 1e3, 4),
        "config": {"workload": shape.name, "T": shape.T, "H": shape.H,
                   "n_routed": shape.n_routed, "n_shared": shape.n_shared,
                   "top_k": shape.top_k, "inter": shape.inter, "gate": shape.gate,
                   "act": shape.act, "parallelism": f"replicas x{world}",
                   "l2": "flushed between timed steps (512 MiB written, then 512 MiB read so the written lines reach HBM before the step)"},
        "expert_ffn_ms": round(ffn_s * 1e3, 4),
        "expert_tflops": round(flops / ffn_s / 1e12, 1),
        "layer_tflops": round(flops / layer_s / 1e12, 1),
        "roofline": roof,
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(u_host.numel() * u_host.element_size()),
                "d2h_bytes_per_step": int(h_host.numel() * h_host.element_size()),
                "api": "moe_layer_forward_host_stream (K steps' batches, copies overlapping "
                       "the neighbouring steps' layers)",
                "per_call": {"value": round(e2e_call_value, 1), "unit": "tokens/s",
                             "api": "moe_layer_forward_host, one call per step"}},
        "gpu_launches": layer.launches_per_step * K,
        "clocks": clk.summary(),
    }
    if graph_entry is not None:
        entry["graph_replay"] = graph_entry
    del u_host, h_host, u_dev, u_slots, h_slots
    return entry, layer


def memory_kernel_bytes(s: W.MoEShape) -> dict:
    """Minimal DRAM bytes of each memory-bound launch of one layer step (the
    inputs read once, the outputs written once; bf16 or fp32 rows)."""
    e = 2 if s.dtype == "bf16" else 4
    T, H, E, k, Ks = s.T, s.H, s.n_routed, s.top_k, s.n_shared
    n_chunks = -(-T // 256)
    return {
        # logits in, bias in; choice and gate weights out
        "route_kernel": T * E * 4 + E * 4 + T * k * 8,
        # choice in, per-chunk histograms out
        "dispatch_count": T * k * 4 + n_chunks * E * 4,
        # histograms in, chunk bases and offsets out
        "dispatch_scan": 2 * n_chunks * E * 4 + (E + 1) * 4,
        # choice and chunk bases in, row_token and slot_row out
        "dispatch_scatter": T * k * 4 + n_chunks * E * 4 + 2 * T * k * 4,
        # every token row read once and written to its k rows; slot rows in
        "scatter_token_rows": T * H * e + T * k * H * e + T * k * 4,
        # routed outputs, shared outputs and u in, h out; slot rows and weights in
        "combine_kernel": (T * k + T * Ks + T) * H * e + T * H * e + T * k * 8,
    }


def run_memory_kernels(args):
    """Times the memory-bound kernels of one layer step (route, dispatch's
    three kernels and row scatter, combine) on a workload's token batch,
    without allocating expert weights: the expert outputs combine reads are
    seeded random rows.  L2 is flushed before every timed launch."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s = W.SHAPES[args.workload]
    peaks, peak_src = load_peaks()
    inp = W.make_token_inputs(s, dev, seed=0)
    T, H, E, k, Ks = s.T, s.H, s.n_routed, s.top_k, s.n_shared
    dt = s.torch_dtype
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    off = torch.empty((E + 1,), dtype=torch.int32, device=dev)
    row_token = torch.empty((T * k,), dtype=torch.int32, device=dev)
    slot_row = torch.empty((T * k,), dtype=torch.int32, device=dev)
    u_perm = torch.empty((T * k, H), dtype=dt, device=dev)
    y_perm = torch.randn((T * k, H), generator=gen, device=dev).to(dt)
    y_shared = torch.randn((Ks, T, H), generator=gen, device=dev).to(dt)
    h = torch.empty((T, H), dtype=dt, device=dev)
    ws = M.alloc_workspace(M.moe_dispatch_workspace_size(s), dev)
    flush = L2Flush(dev)
    steps = {
        "router_logits": lambda: M.moe_router_logits(s, inp["u"], inp["centroids"],
                                                     inp["logit_offset"], logits),
        "route": lambda: M.moe_route(s, logits, inp["select_bias"], idx, w),
        "dispatch": lambda: M.moe_dispatch(s, idx, inp["u"], off, row_token, slot_row, u_perm,
                                           ws),
        "combine": lambda: M.moe_combine(s, inp["u"], y_perm, y_shared, w, slot_row, h),
    }
    for _ in range(args.warmup):
        for f in steps.values():
            f()
    torch.cuda.synchronize()
    ms = {n: [] for n in steps}
    for _ in range(args.steps):
        for n, f in steps.items():
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            f()
            b.record()
            ms[n].append((a, b))
    torch.cuda.synchronize()
    st, code = M.moe_device_status()
    if st != M.MOE_OK:
        raise RuntimeError(f"device status {st} code {code}")
    alg = memory_kernel_bytes(s)
    call_bytes = {"route": alg["route_kernel"],
                  "dispatch": sum(alg[n] for n in ("dispatch_count", "dispatch_scan",
                                                   "dispatch_scatter", "scatter_token_rows")),
                  "combine": alg["combine_kernel"],
                  "router_logits": T * H * (2 if s.dtype == "bf16" else 4)
                  + E * H * (2 if s.dtype == "bf16" else 4) + T * E * 4}
    out = {}
    for n, evs in ms.items():
        t = statistics.median(a.elapsed_time(b) for a, b in evs) / 1e3
        gb = call_bytes[n] / t / 1e9
        out[n] = {"us": round(t * 1e6, 2), "algorithmic_bytes": call_bytes[n],
                  "gbs": round(gb, 1), "frac_of_hbm": round(gb / peaks["hbm_gbs"], 4)}
    print(json.dumps({"mode": "memory_kernels", "workload": s.name, "steps": args.steps,
                      "peak_hbm_gbs": peaks["hbm_gbs"], "peak_source": peak_src,
                      "per_kernel_bytes": alg, "calls": out,
                      "note": "median of CUDA-event times per C-ABI call, L2 flushed before "
                              "each; dispatch is four kernels (count, scan, scatter, row "
                              "scatter)"}),
          flush=True)


def run_cuda(args):
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks, peak_src = load_peaks()
    peaks = dict(peaks, _source=peak_src)
    flush = L2Flush(dev)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()

    names = [args.workload]
    if not args.only:
        names += [n for n in EXTRA_WORKLOADS if n != args.workload]
    entries = {}
    cpu = None
    for n, name in enumerate(names):
        shape = W.SHAPES[name]
        entry, layer = measure_forward(args, shape, dev, flush, world, peaks, barrier)
        if not args.no_backward and (name == BACKWARD_WORKLOAD or
                                     (args.backward and name == args.workload)):
            entry["backward"] = measure_backward(args, shape, layer, flush, dev, peaks)
        if n == 0 and rank == 0 and world == 1 and not args.no_cpu_baseline:
            cpu = cpu_baseline(shape, layer, args.cpu_sample)
        entries[name] = entry
        del layer
        torch.cuda.empty_cache()

    head = entries[args.workload]
    shape = W.SHAPES[args.workload]
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if shape.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) tokens, N(0,1/fan_in) weights)",
        "config": head["config"],
        "expert_ffn_ms": head["expert_ffn_ms"], "expert_tflops": head["expert_tflops"],
        "layer_tflops": head["layer_tflops"],
        "roofline": head["roofline"], "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"], "clocks": head["clocks"],
        "peaks_note": PEAK_NOTE,
    }
    if "backward" in head:
        line["backward"] = head["backward"]
    if cpu is not None:
        line["cpu_baseline"] = cpu
    line["workloads"] = {k: v for k, v in entries.items() if k != args.workload}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------------ CPU oracle legs

# float64 copies of all expert weights are kept only up to this size; larger
# layers convert each expert's stored weights when the oracle asks for them
F64_CACHE_BYTES = 8 << 30


def f64_weight_bytes(shape) -> int:
    return (shape.n_routed + shape.n_shared) * shape.n_mats * shape.H * shape.inter * 8


def _oracle_setup(shape, inp):
    """What the oracle needs, as host float64 arrays.  Returns (O, routed_fn,
    shared_fn, centroids, offsets, bias, cached): with cached, every expert's
    weights are converted once and kept; otherwise each call converts the
    stored weights again (the caller decides whether that is timed)."""
    import oracle.moe_oracle as O  # the oracle is imported only for this leg
    # copied to the host in the stored type, widened there (exact for bf16)
    np64 = lambda t: t.detach().cpu().to(torch.float64).numpy()
    cached = f64_weight_bytes(shape) <= F64_CACHE_BYTES
    routed = {}

    def convert(w1, w3, w2, j):
        return (np64(w1[j]), None if w3 is None else np64(w3[j]), np64(w2[j]))

    def routed_fn(e):
        if not cached:
            return convert(inp.w1, inp.w3, inp.w2, e)
        if e not in routed:
            routed[e] = convert(inp.w1, inp.w3, inp.w2, e)
        return routed[e]

    shared = [convert(inp.sw1, inp.sw3, inp.sw2, j) for j in range(shape.n_shared)]
    cents = np64(inp.centroids)
    off = None if inp.logit_offset is None else np64(inp.logit_offset)
    bias = None if inp.select_bias is None else inp.select_bias.cpu().numpy()
    return O, routed_fn, (lambda j: shared[j]), cents, off, bias, cached


def _oracle_tokens(O, shape, u_rows, routed_fn, shared_fn, cents, off, bias):
    z = O.router_logits(u_rows, cents, off)
    r = O.route(z, shape.gate, shape.top_k, bias)
    O.dispatch(r["idx"], shape.n_routed)
    return O.layer_forward(u_rows, r, routed_fn, shared_fn, shape.n_shared, shape.act)


def _preconvert(O, shape, u, routed_fn, cents, off, bias):
    z = O.router_logits(u, cents, off)
    for e in np.unique(O.route(z, shape.gate, shape.top_k, bias)["idx"]):
        routed_fn(int(e))


def _threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return len(os.sched_getaffinity(0))


def _weights_note(shape, cached):
    if cached:
        return "expert weights converted to float64 once, outside the timing"
    return (f"each used expert's stored bf16 weights converted to float64 inside the timing "
            f"(float64 copies of all {shape.n_routed + shape.n_shared} experts would take "
            f"{f64_weight_bytes(shape) / 2**30:.0f} GiB of host memory)")


def cpu_baseline(shape, layer, n_sample, min_seconds=10.0):
    """The oracle on bounded samples of the workload's tokens, repeated until
    about ``min_seconds`` of CPU work; tokens/s over all repetitions."""
    inp = layer.inp
    O, routed_fn, shared_fn, cents, off, bias, cached = _oracle_setup(shape, inp)
    rng = np.random.default_rng(0)
    # a layer whose float64 weights cannot stay cached converts every used
    # expert per sample: fewer tokens keep the leg within ~10-30 s
    n = min(n_sample if cached else max(1, n_sample // 4), shape.T)
    done, elapsed, reps = 0, 0.0, 0
    while elapsed < min_seconds and reps < 64:
        rows = np.sort(rng.choice(shape.T, size=n, replace=False))
        u = inp.u[torch.from_numpy(rows).to(inp.u.device)].to(torch.float64).cpu().numpy()
        if cached:
            _preconvert(O, shape, u, routed_fn, cents, off, bias)
        t0 = time.perf_counter()
        _oracle_tokens(O, shape, u, routed_fn, shared_fn, cents, off, bias)
        elapsed += time.perf_counter() - t0
        done += n
        reps += 1
    return {"value": round(done / elapsed, 2), "unit": "tokens/s", "cores": _threads(),
            "kind": "oracle", "sample": f"{reps} x {n} random tokens of {shape.name} "
            f"(T={shape.T}): full layer (logits, route, dispatch, FFN, combine) in float64 "
            f"NumPy; {_weights_note(shape, cached)}; {elapsed:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    shape = W.SHAPES[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = W.make_inputs(shape, dev, seed=0)
    O, routed_fn, shared_fn, cents, off, bias, cached = _oracle_setup(shape, inp)
    u_all = inp.u
    n = args.ref_sample or (256 if cached else 8)
    n = min(n, shape.T)
    rng = np.random.default_rng(1)
    samples = []
    for _ in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(shape.T, size=n, replace=False))
        samples.append(u_all[torch.from_numpy(rows).to(u_all.device)].to(torch.float64).cpu().numpy())
    if cached:              # expert weights resident in host memory before timing
        for u in samples:
            _preconvert(O, shape, u, routed_fn, cents, off, bias)
    for u in samples[:args.warmup]:
        _oracle_tokens(O, shape, u, routed_fn, shared_fn, cents, off, bias)
    t0 = time.perf_counter()
    for u in samples[args.warmup:]:
        _oracle_tokens(O, shape, u, routed_fn, shared_fn, cents, off, bias)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": shape.name, "T": shape.T, "H": shape.H,
                   "n_routed": shape.n_routed, "n_shared": shape.n_shared,
                   "top_k": shape.top_k, "inter": shape.inter, "gate": shape.gate,
                   "act": shape.act},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": _threads(),
                         "kind": "oracle",
                         "sample": f"{n} random tokens per step of {shape.name} "
                                   f"(T={shape.T}); {_weights_note(shape, cached)}"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def relaunch_under_torchrun(n: int):
    """Re-execute this script as n torchrun processes on this node."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1", "--master-port",
           str(port), os.path.abspath(__file__), *sys.argv[1:]]
    os.execv(sys.executable, cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.SHAPES))
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--cpu-sample", type=int, default=256,
                    help="tokens per sample of the cpu_baseline leg")
    ap.add_argument("--ref-sample", type=int, default=0,
                    help="tokens per step of --impl reference (0: 256 when the float64 "
                         "weights fit the host cache, else 8)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the timed moe_layer_backward leg")
    ap.add_argument("--backward", action="store_true",
                    help="time moe_layer_backward on the chosen workload too (by default "
                         "only the DeepSeekMoE-16B-shaped workload gets the backward leg)")
    ap.add_argument("--only", action="store_true",
                    help="time the chosen workload only, not the extra ones")
    ap.add_argument("--memory-kernels", action="store_true",
                    help="time the memory-bound kernels of the chosen workload's step "
                         "(no expert weights are allocated)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    _, world, _ = dist_env()
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        relaunch_under_torchrun(args.gpus)
    if world != args.gpus:
        sys.exit(f"bench.py: --gpus {args.gpus} does not match WORLD_SIZE={world}")
    if args.impl == "reference":
        run_reference(args)
    elif args.memory_kernels:
        run_memory_kernels(args)
    else:
        run_cuda(args)


if __name__ == "__main__":
    main()
