"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding, run the oracle on the same seeded inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle.moe_oracle as O
from fine_grained_shared_gemm_b300 import moe as M
from fine_grained_shared_gemm_b300 import workloads as W

NEAR_TIE = 1e-5            # k-th vs (k+1)-th score/key gap below which a choice may differ
TOL = {"f32": 1e-4, "bf16": 2e-2}   # max|Δ| ≤ TOL · max|ref| on layer and FFN outputs


def np64(t: torch.Tensor) -> np.ndarray:
    """float64 copy on the host (copied in the stored type, widened there)."""
    return t.detach().cpu().to(torch.float64).numpy()


def expert_fns(inp: W.MoEInputs):
    """Oracle weight accessors: fetch one expert at a time as float64."""
    def routed(e):
        return (np64(inp.w1[e]), None if inp.w3 is None else np64(inp.w3[e]), np64(inp.w2[e]))

    def shared(j):
        return (np64(inp.sw1[j]), None if inp.sw3 is None else np64(inp.sw3[j]), np64(inp.sw2[j]))
    return routed, shared


def bias_np(inp: W.MoEInputs):
    return None if inp.select_bias is None else inp.select_bias.cpu().numpy()


def oracle_route(shape: W.MoEShape, logits_np, inp: W.MoEInputs):
    r = O.route(logits_np, shape.gate, shape.top_k,
                bias_np(inp) if shape.gate == W.GATE_SIGMOID_BIAS else None,
                shape.n_groups, shape.topk_groups)
    # a near-tie of the last kept group counts like one of the k-th expert
    r["gap"] = np.minimum(r["gap"], r["group_gap"])
    return r


def gpu_route(shape, logits: torch.Tensor, bias):
    T, k = shape.T, shape.top_k
    dev = logits.device
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    gap = torch.empty((T,), dtype=torch.float32, device=dev)
    M.moe_route(shape, logits, bias, idx, w, gap)
    return idx, w, gap


def compare_routing(shape, gpu_idx, gpu_w, ref):
    """Choices equal except on near-ties (reported, not failed); weights of the
    equal rows within 1e-6 + 1e-5·|g|.  Returns the near-tie row mask."""
    gi = gpu_idx.cpu().numpy().astype(np.int64)
    gw = gpu_w.cpu().numpy().astype(np.float64)
    diff = np.any(gi != ref["idx"], axis=1)
    near = ref["gap"] < NEAR_TIE
    bad = diff & ~near
    assert not bad.any(), (
        f"{int(bad.sum())} rows choose different experts without a near-tie; first "
        f"{np.nonzero(bad)[0][:5]} gpu={gi[bad][:2]} ref={ref['idx'][bad][:2]}")
    same = ~diff
    err = np.abs(gw[same] - ref["weights"][same])
    lim = 1e-6 + 1e-5 * np.abs(ref["weights"][same])
    assert np.all(err <= lim), f"gate weights off by {float((err - lim).max())} over the limit"
    return diff


def route_with_choice(shape, ref, idx):
    """Oracle gate weights for a given choice (used where a near-tie flipped it)."""
    s = ref["scores"]
    g = np.take_along_axis(s, idx, axis=1)
    if shape.gate == W.GATE_SIGMOID_BIAS and idx.shape[1]:
        g = g / g.sum(axis=1, keepdims=True)
    return dict(idx=idx, weights=g)


def assert_close(got: np.ndarray, ref: np.ndarray, tol: float, what: str):
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    assert err <= tol * max(scale, 1e-30), f"{what}: max|Δ| = {err:.3e} > {tol} · {scale:.3e}"
    return err, scale


def layer_buffers(shape, device):
    ws = M.alloc_workspace(M.moe_layer_workspace_size(shape), device)
    h = torch.empty((shape.T, shape.H), dtype=shape.torch_dtype, device=device)
    return ws, h
