"""Benchmark of the DeepSeekMoE layer forward on B300.

One step = one pass of the whole layer (router logits, route, dispatch,
expert FFNs, combine) over one batch of T seeded synthetic tokens whose
inputs are already resident in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the same workload

Under torchrun every rank runs an independent replica of the layer on its own
GPU (tokens are independent, so the layer shards by batch with no exchange);
value = all tokens processed / the slowest rank's time.
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

DEFAULT_WORKLOAD = "dsmoe16b_bf16"
METRIC = "MoE layer tokens/s & TFLOP/s (% bf16 peak); decode weight GB/s (% HBM)"
L2_FLUSH_BYTES = 512 << 20     # larger than the 126 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


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


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


def expert_flops(s: W.MoEShape) -> int:
    return s.T * (s.top_k + s.n_shared) * s.n_mats * 2 * s.H * s.inter


def touched_weight_bytes(s: W.MoEShape, offsets: np.ndarray) -> int:
    """Expert weights a step must read at least once: every expert with a token."""
    used = int((np.diff(offsets) > 0).sum()) + s.n_shared
    return used * s.n_mats * s.H * s.inter * 2 + s.n_routed * s.H * 2


def ffn_alg_bytes(s: W.MoEShape, offsets: np.ndarray) -> int:
    """Bytes one moe_expert_ffn call must move at least: every expert with a
    token reads its weights once; the expert input rows come in (the permuted
    rows, and u once per shared expert), the activation goes out and back
    in, the outputs go out."""
    e = 2 if s.dtype == "bf16" else 4
    used = int((np.diff(offsets) > 0).sum()) + s.n_shared
    rows = s.T * (s.top_k + s.n_shared)
    return (used * s.n_mats * s.H * s.inter + rows * s.H * 2 + rows * s.inter * 2) * e


def ffn_roofline(shape: W.MoEShape, offsets: np.ndarray, ffn_s: float, peaks: dict) -> dict:
    """The expert FFN's roofline entry for one launch of ffn_s seconds.

    Decode-shaped layers (T·k < 2E) are timed against the HBM copy bandwidth
    with the weights of every touched expert as the algorithmic bytes.  Other
    layers are timed against their binding roof: the larger of the two lower
    bounds, algorithmic FLOPs at the measured tensor peak and algorithmic
    bytes at the measured copy bandwidth (the V3-shaped layer sits just on the
    memory side of the ridge); the other roof is reported under other_roof.
    """
    flops = expert_flops(shape)
    if shape.T * shape.top_k < 2 * shape.n_routed:
        gb = touched_weight_bytes(shape, offsets) / ffn_s / 1e9
        return {"bound": "hbm", "achieved": round(gb, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(gb / peaks["hbm_gbs"], 4)}
    alg_bytes = ffn_alg_bytes(shape, offsets)
    t_flops = flops / (peaks["bf16_tflops"] * 1e12)
    t_bytes = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    tf = flops / ffn_s / 1e12
    gb = alg_bytes / ffn_s / 1e9
    tensor = {"bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_tflops"],
              "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4)}
    memory = {"bound": "hbm", "achieved": round(gb, 1), "peak": peaks["hbm_gbs"],
              "unit": "GB/s", "frac": round(gb / peaks["hbm_gbs"], 4),
              "algorithmic_bytes": alg_bytes}
    roof, other = (memory, tensor) if t_bytes > t_flops else (tensor, memory)
    return dict(roof, other_roof=other)


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
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples)}


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
        self.launches_per_step = 10

    def step(self, ev=None):
        s, i = self.s, self.inp
        M.moe_router_logits(s, i.u, i.centroids, i.logit_offset, self.logits)
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
    n += 2 if k else 0                            # gather dh rows, row gate weights
    n += 2                                        # FFN plan, weight-gradient plan
    n += 1 if rows else 0                         # dm = dh W2
    n += s.n_shared + (1 if k else 0)             # activation derivative
    n += 1 + 3                                    # gate, router GEMMs + u transpose
    n += (1 if rows else 0) + 1                   # dx, du
    n += 1 + (2 if k else 0)                      # dh and routed x, dh transposes
    n += 2                                        # weight-gradient GEMMs
    return n


def forward_launches(s: W.MoEShape) -> int:
    """Kernel launches of one moe_layer_forward(_train) call."""
    return 10 if s.top_k > 0 else 7


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
    for i in range(K):
        flush.zero_()
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
    for i in range(K):
        flush.zero_()
        ev_f[i][0].record()
        M.moe_layer_forward_train(s, layer.wt, inp.u, h, saved, layer.ws_l)
        ev_f[i][1].record()
        flush.zero_()
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
    del ws, g, grads, saved
    return {"tokens_per_s": round(s.T / (ms / 1e3), 1), "ms_per_step": round(ms, 4),
            "algorithmic_tflop": round(flops / 1e12, 4), "tflops": round(tf, 1),
            "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
            "gpu_launches": backward_launches(s) * K,
            "note": "recomputes routing and the gate/up pre-activations from u; "
                    "weight gradients fp32",
            "training_step": {
                "forward_train_ms": round(f_ms, 4), "backward_saved_ms": round(b_ms, 4),
                "gpu_launches": (forward_launches(s) + backward_launches(s, saved=True)) * K,
                "tokens_per_s": round(s.T / ((f_ms + b_ms) / 1e3), 1),
                "tflops": round(step_flops / ((f_ms + b_ms) / 1e3) / 1e12, 1),
                "note": "moe_layer_forward_train + moe_layer_backward on its saved tensors"}}


def run_cuda(args):
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    shape = W.SHAPES[args.workload]
    layer = Layer(shape, dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        layer.step()
    st, code = M.moe_device_status()
    if st != M.MOE_OK:
        raise RuntimeError(f"device status {st} code {code} after warm-up")

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ffn_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
    barrier()
    with ClockSampler(dev) as clk:
        for i in range(K):
            flush.zero_()                       # L2 flushed between timed steps
            starts[i].record()
            layer.step(ffn_ev[i])
            ends[i].record()
        barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ffn_ms = [a.elapsed_time(b) for a, b in ffn_ev]
    total_s = max_over_ranks(sum(step_ms) / 1e3, dev)
    tokens = shape.T * K * world
    value = tokens / total_s

    # end to end through the host-buffer entry point: H2D of u, layer, D2H of h
    u_host = layer.inp.u.cpu().pin_memory()
    h_host = torch.empty_like(u_host).pin_memory()
    u_dev = torch.empty_like(layer.inp.u)
    for _ in range(max(1, args.warmup)):
        M.moe_layer_forward_host(shape, layer.wt, u_host, h_host, u_dev, layer.h, layer.ws_l)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        M.moe_layer_forward_host(shape, layer.wt, u_host, h_host, u_dev, layer.h, layer.ws_l)
    e1.record()
    barrier()
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, dev)
    st, code = M.moe_device_status()
    if st != M.MOE_OK:
        raise RuntimeError(f"device status {st} code {code}")

    peaks, peak_src = load_peaks()
    ffn_avg_s = sum(ffn_ms) / len(ffn_ms) / 1e3
    flops = expert_flops(shape)
    offsets = layer.off.cpu().numpy()
    roof = ffn_roofline(shape, offsets, ffn_avg_s, peaks)
    roof.update({"traffic": recorded_traffic(args.workload), "kernel": "moe_expert_ffn",
                 "peak_source": f"{peak_src} (burst)", "ms_per_launch": round(ffn_avg_s * 1e3, 4)})

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(total_s / K * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
        if shape.dtype == "bf16" else "f32", "data": "synthetic (seeded N(0,1) tokens, "
        "N(0,1/fan_in) weights)",
        "config": {"workload": shape.name, "T": shape.T, "H": shape.H,
                   "n_routed": shape.n_routed, "n_shared": shape.n_shared,
                   "top_k": shape.top_k, "inter": shape.inter, "gate": shape.gate,
                   "act": shape.act, "parallelism": f"replicas x{world}",
                   "l2": "flushed between timed steps (512 MiB write)"},
        "expert_tflops": round(flops / ffn_avg_s / 1e12, 1),
        "layer_tflops": round(flops / (total_s / K / world) / 1e12, 1) if world == 1 else None,
        "roofline": roof,
        "e2e": {"value": round(tokens / e2e_s, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(u_host.numel() * u_host.element_size()),
                "d2h_bytes_per_step": int(h_host.numel() * h_host.element_size())},
        "gpu_launches": layer.launches_per_step * K,
        "clocks": clk.summary(),
    }
    if not args.no_backward:
        line["backward"] = measure_backward(args, shape, layer, flush, dev, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(shape, layer, args.cpu_sample)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------------ CPU oracle legs

def _oracle_setup(shape, inp):
    """Host float64 copies of what the oracle needs (outside any timing)."""
    import oracle.moe_oracle as O  # the oracle is imported only for this leg
    np64 = lambda t: t.detach().to(torch.float64).cpu().numpy()
    routed = {}
    shared = [(np64(inp.sw1[j]), None if inp.sw3 is None else np64(inp.sw3[j]),
               np64(inp.sw2[j])) for j in range(shape.n_shared)]

    def routed_fn(e):
        if e not in routed:
            routed[e] = (np64(inp.w1[e]), None if inp.w3 is None else np64(inp.w3[e]),
                         np64(inp.w2[e]))
        return routed[e]
    cents = np64(inp.centroids)
    off = None if inp.logit_offset is None else np64(inp.logit_offset)
    bias = None if inp.select_bias is None else inp.select_bias.cpu().numpy()
    return O, routed_fn, (lambda j: shared[j]), cents, off, bias


def _oracle_tokens(O, shape, u_rows, routed_fn, shared_fn, cents, off, bias):
    z = O.router_logits(u_rows, cents, off)
    r = O.route(z, shape.gate, shape.top_k, bias)
    O.dispatch(r["idx"], shape.n_routed)
    return O.layer_forward(u_rows, r, routed_fn, shared_fn, shape.n_shared, shape.act)


def _threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return len(os.sched_getaffinity(0))


def cpu_baseline(shape, layer, n_sample, min_seconds=10.0):
    """The oracle on bounded samples of the workload's tokens, repeated until
    about ``min_seconds`` of CPU work; tokens/s over all repetitions."""
    inp = layer.inp
    O, routed_fn, shared_fn, cents, off, bias = _oracle_setup(shape, inp)
    rng = np.random.default_rng(0)
    n = min(n_sample, shape.T)
    done, elapsed, reps = 0, 0.0, 0
    while elapsed < min_seconds and reps < 64:
        rows = np.sort(rng.choice(shape.T, size=n, replace=False))
        u = inp.u[torch.from_numpy(rows).to(inp.u.device)].to(torch.float64).cpu().numpy()
        # weights of every expert these tokens use are converted before timing
        z = O.router_logits(u, cents, off)
        for e in np.unique(O.route(z, shape.gate, shape.top_k, bias)["idx"]):
            routed_fn(int(e))
        t0 = time.perf_counter()
        _oracle_tokens(O, shape, u, routed_fn, shared_fn, cents, off, bias)
        elapsed += time.perf_counter() - t0
        done += n
        reps += 1
    return {"value": round(done / elapsed, 2), "unit": "tokens/s", "cores": _threads(),
            "kind": "oracle", "sample": f"{reps} x {n} random tokens of {shape.name} "
            f"(T={shape.T}): full layer (logits, route, dispatch, FFN, combine) in float64 "
            f"NumPy, weights pre-converted to float64 outside the timing; {elapsed:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    shape = W.SHAPES[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = W.make_inputs(shape, dev, seed=0)
    O, routed_fn, shared_fn, cents, off, bias = _oracle_setup(shape, inp)
    u_all = inp.u
    n = min(args.cpu_sample, shape.T)
    rng = np.random.default_rng(1)
    samples = []
    for _ in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(shape.T, size=n, replace=False))
        samples.append(u_all[torch.from_numpy(rows).to(u_all.device)].to(torch.float64).cpu().numpy())
    for u in samples:       # expert weights resident in host memory before timing
        z = O.router_logits(u, cents, off)
        for e in np.unique(O.route(z, shape.gate, shape.top_k, bias)["idx"]):
            routed_fn(int(e))
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
                   "top_k": shape.top_k, "inter": shape.inter},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": _threads(),
                         "kind": "oracle", "sample": f"{n} tokens per step of {shape.name}"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.SHAPES))
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--cpu-sample", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the timed moe_layer_backward leg")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_cuda(args)


if __name__ == "__main__":
    main()
