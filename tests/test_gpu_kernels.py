"""GPU parity of each step of the layer against the oracle, on seeded inputs
of several tiles with ragged tails, plus the edge cases of the method."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from fine_grained_shared_gemm_b300 import moe as M
from fine_grained_shared_gemm_b300 import workloads as W
from parity_helpers import (TOL, assert_close, bias_np, compare_routing, expert_fns,
                            gpu_route, np64, oracle_route)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def S(name, **kw):
    base = dict(T=300, H=256, n_routed=8, n_shared=1, top_k=2, inter=128,
                gate=W.GATE_SOFTMAX, act=W.ACT_SWIGLU, dtype="bf16")
    base.update(kw)
    return W.MoEShape(name=name, **base)


# ---------------------------------------------------------------- routing

ROUTE_CASES = [
    # (E, k, gate, kind)
    (14, 6, W.GATE_SOFTMAX, "normal"),
    (64, 6, W.GATE_SOFTMAX, "normal"),
    (63, 7, W.GATE_SOFTMAX, "normal"),
    (256, 32, W.GATE_SOFTMAX, "normal"),
    (16, 2, W.GATE_SOFTMAX, "ties"),
    (40, 5, W.GATE_SOFTMAX, "skewed"),
    (256, 8, W.GATE_SIGMOID_BIAS, "normal"),
    (384, 8, W.GATE_SIGMOID_BIAS, "skewed"),
    (33, 3, W.GATE_SIGMOID_BIAS, "ties"),
    (8, 8, W.GATE_SOFTMAX, "normal"),      # k = E
    (1, 1, W.GATE_SOFTMAX, "normal"),      # single expert, g = 1
    (32, 1, W.GATE_SIGMOID_BIAS, "normal"),  # top-1: weight 1
    (1000, 4, W.GATE_SOFTMAX, "normal"),   # widest router
]


@pytest.mark.parametrize("E,k,gate,kind", ROUTE_CASES)
def test_route_bit_exact_from_same_logits(E, k, gate, kind):
    T = 1001
    shape = S("route", T=T, n_routed=E, top_k=k, gate=gate)
    z = W.random_logits(T, E, seed=E * 31 + k, kind=kind)
    bias = None
    if gate == W.GATE_SIGMOID_BIAS:
        g = torch.Generator().manual_seed(E)
        bias = (torch.rand(E, generator=g) * 0.2 - 0.1)
    ref = O.route(z.numpy(), gate, k, None if bias is None else bias.numpy())
    idx, w, gap = gpu_route(shape, z.to(DEV), None if bias is None else bias.to(DEV))
    diff = compare_routing(shape, idx, w, ref)
    if kind == "ties" and gate == W.GATE_SOFTMAX:
        assert not diff.any()     # exact ties are decided by index on both sides
    g = gap.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref["gap"])
    assert np.array_equal(np.isfinite(g), fin)
    assert np.all(np.abs(g[fin] - ref["gap"][fin]) <= 1e-6 + 1e-5 * np.abs(ref["gap"][fin]))


GROUP_CASES = [
    # (E, k, n_groups, topk_groups, gate, kind)
    (256, 8, 8, 4, W.GATE_SIGMOID_BIAS, "normal"),   # the V3 setting: 8 groups, 4 kept
    (64, 6, 4, 2, W.GATE_SOFTMAX, "normal"),
    (64, 8, 8, 2, W.GATE_SIGMOID_BIAS, "skewed"),    # exactly k experts in the kept groups
    (96, 6, 32, 6, W.GATE_SOFTMAX, "skewed"),        # 32 groups of 3
    (16, 2, 4, 1, W.GATE_SOFTMAX, "ties"),           # integer logits: exact group ties
    (40, 5, 5, 5, W.GATE_SIGMOID_BIAS, "normal"),    # every group kept = no limit
    (384, 8, 32, 4, W.GATE_SIGMOID_BIAS, "normal"),
]


@pytest.mark.parametrize("E,k,G,M,gate,kind", GROUP_CASES)
def test_group_limited_route_bit_exact_from_same_logits(E, k, G, M, gate, kind):
    """Group-limited routing (page "02 · 细粒度 MoE", §4): the choice equals the
    oracle's from the same fp32 logits except where the last kept group or the
    k-th expert wins by less than 1e-5 (reported, not failed)."""
    T = 1001
    shape = S("groups", T=T, n_routed=E, top_k=k, gate=gate, n_groups=G, topk_groups=M)
    z = W.random_logits(T, E, seed=E * 7 + G, kind=kind)
    bias = None
    if gate == W.GATE_SIGMOID_BIAS:
        g = torch.Generator().manual_seed(E + G)
        bias = (torch.rand(E, generator=g) * 0.2 - 0.1)
    ref = O.route(z.numpy(), gate, k, None if bias is None else bias.numpy(), G, M)
    idx, w, gap = gpu_route(shape, z.to(DEV), None if bias is None else bias.to(DEV))
    near = dict(ref)
    near["gap"] = np.minimum(ref["gap"], ref["group_gap"])
    diff = compare_routing(shape, idx, w, near)
    gi = idx.cpu().numpy()
    gsize = E // G
    # every chosen expert lies in a kept group: at most M distinct groups per token
    assert max(len(set((gi[t] // gsize).tolist())) for t in range(T)) <= M
    if kind == "ties":
        assert not diff.any()     # exact group and expert ties go to the lower index on both sides
    g = gap.cpu().numpy().astype(np.float64)
    same = ~diff
    fin = np.isfinite(ref["gap"]) & same
    assert np.array_equal(np.isfinite(g)[same], np.isfinite(ref["gap"])[same])
    assert np.all(np.abs(g[fin] - ref["gap"][fin]) <= 1e-6 + 1e-5 * np.abs(ref["gap"][fin]))
    print(f"E={E} G={G} M={M}: {int(diff.sum())} near-tie flips")


def test_route_zero_tokens_and_zero_k():
    shape = S("empty", T=0, n_routed=8, top_k=2)
    z = torch.empty((0, 8), device=DEV)
    gpu_route(shape, z, None)
    shape = S("k0", T=5, n_routed=8, top_k=0)
    idx, w, gap = gpu_route(shape, torch.randn(5, 8, device=DEV), None)
    torch.cuda.synchronize()


# ---------------------------------------------------------------- logits

@pytest.mark.parametrize("shape", [
    S("lg_f32", T=257, H=256, n_routed=14, dtype="f32", act=W.ACT_RELU),
    S("lg_bf16", T=300, H=512, n_routed=64),
    S("lg_bf16_wide", T=1030, H=2048, n_routed=256),
    S("lg_bf16_odd", T=77, H=1024, n_routed=63),
    S("lg_bf16_decode", T=64, H=7168, n_routed=384, gate=W.GATE_SIGMOID_BIAS, logit_offset_std=1.0),
], ids=lambda s: s.name)
def test_router_logits(shape):
    inp = W.make_inputs(shape, DEV, seed=3)
    u, e = np64(inp.u), np64(inp.centroids)
    off = None if inp.logit_offset is None else np64(inp.logit_offset)
    ref = O.router_logits(u, e, off).astype(np.float64)
    # fp32 accumulation of H products: bounded by a small multiple of Σ|u_d e_d|
    bound = 1e-5 * (np.abs(u) @ np.abs(e).T) + 1e-6
    # the contraction whole (no workspace), and with the workspace, which cuts
    # it into ranges for few-tile batches (the decode shape: 28 ranges)
    need = M.moe_router_logits_workspace_size(shape)
    if shape.name == "lg_bf16_decode":
        assert need == 28 * shape.T * shape.n_routed * 4
    outs = []
    for ws in (None, M.alloc_workspace(need, DEV)):
        logits = torch.full((shape.T, shape.n_routed), float("nan"), dtype=torch.float32,
                            device=DEV)
        M.moe_router_logits(shape, inp.u, inp.centroids, inp.logit_offset, logits, ws)
        got = logits.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) - bound))
        outs.append(got)
        if ws is not None:   # the ranges are added in a fixed order: the same on every run
            M.moe_router_logits(shape, inp.u, inp.centroids, inp.logit_offset, logits, ws)
            assert np.array_equal(logits.cpu().numpy().astype(np.float64), got)
    if need == 0:
        assert np.array_equal(outs[0], outs[1])


def test_router_logits_rejects_a_short_workspace():
    shape = S("lg_short_ws", T=64, H=1024, n_routed=64)
    need = M.moe_router_logits_workspace_size(shape)
    assert need > 0
    inp = W.make_inputs(shape, DEV, seed=3)
    logits = torch.empty((shape.T, shape.n_routed), dtype=torch.float32, device=DEV)
    st = M.lib().moe_router_logits(M.ctypes.byref(M.shape_struct(shape)), M._ptr(inp.u),
                                   M._ptr(inp.centroids), None, M._ptr(logits),
                                   M._ptr(M.alloc_workspace(need, DEV)), need - 16, None)
    assert st == M.MOE_ERR_WORKSPACE
    assert M.moe_device_status() == (M.MOE_OK, 0)


# ---------------------------------------------------------------- dispatch

def _idx_for(shape, seed, kind="normal"):
    z = W.random_logits(shape.T, shape.n_routed, seed=seed, kind=kind).numpy()
    return O.route(z, W.GATE_SOFTMAX, shape.top_k)["idx"]


def _gpu_dispatch(shape, idx_np, u):
    T, k, E = shape.T, shape.top_k, shape.n_routed
    idx = torch.from_numpy(idx_np.astype(np.int32)).to(DEV)
    off = torch.full((E + 1,), -7, dtype=torch.int32, device=DEV)
    row_token = torch.empty(T * k, dtype=torch.int32, device=DEV)
    slot_row = torch.empty(T * k, dtype=torch.int32, device=DEV)
    u_perm = torch.empty((T * k, shape.H), dtype=u.dtype, device=DEV)
    ws = M.alloc_workspace(M.moe_dispatch_workspace_size(shape), DEV)
    M.moe_dispatch(shape, idx, u, off, row_token, slot_row, u_perm, ws)
    return off, row_token, slot_row, u_perm


@pytest.mark.parametrize("T,E,k,kind", [
    (1000, 14, 6, "normal"), (257, 64, 6, "skewed"), (4097, 256, 8, "normal"),
    (513, 384, 8, "skewed"), (300, 8, 8, "normal"), (1, 16, 3, "normal"),
    (700, 40, 1, "skewed"), (2000, 256, 32, "normal"),
])
def test_dispatch_bit_exact(T, E, k, kind):
    shape = S("disp", T=T, n_routed=E, top_k=k)
    idx = _idx_for(shape, seed=T + E, kind=kind)
    u = torch.randn((T, shape.H), device=DEV).to(torch.bfloat16)
    off, row_token, slot_row, u_perm = _gpu_dispatch(shape, idx, u)
    ref = O.dispatch(idx, E)
    assert np.array_equal(off.cpu().numpy(), ref["offsets"])
    assert np.array_equal(row_token.cpu().numpy(), ref["row_token"])
    assert np.array_equal(slot_row.cpu().numpy().reshape(T, k), ref["slot_row"])
    assert torch.equal(u_perm, u[row_token.long()])
    if kind == "skewed":
        assert (ref["counts"] == 0).any() or E <= 8   # some experts receive no token


@pytest.mark.parametrize("T,E,k,H", [
    (1000, 64, 6, 2176),   # 272 vectors a row in segments of 96, 96, 80
    (64, 384, 8, 7168),    # decode-sized: 28 segments of 32 vectors a row
    (3000, 32, 4, 1024),   # one segment a row (enough tokens)
])
def test_dispatch_row_segments(T, E, k, H):
    # the row scatter splits each token row across several warps for small
    # batches; every copy must still land whole
    shape = S("disp_seg", T=T, H=H, n_routed=E, top_k=k)
    idx = _idx_for(shape, seed=T + H)
    u = torch.randn((T, H), device=DEV).to(torch.bfloat16)
    off, row_token, slot_row, u_perm = _gpu_dispatch(shape, idx, u)
    ref = O.dispatch(idx, E)
    assert np.array_equal(row_token.cpu().numpy(), ref["row_token"])
    assert torch.equal(u_perm, u[row_token.long()])


def test_dispatch_all_tokens_to_same_experts():
    T, E, k = 777, 32, 4
    shape = S("hot", T=T, n_routed=E, top_k=k)
    idx = np.tile(np.array([5, 0, 31, 7]), (T, 1))
    u = torch.randn((T, shape.H), device=DEV).to(torch.bfloat16)
    off, row_token, slot_row, u_perm = _gpu_dispatch(shape, idx, u)
    ref = O.dispatch(idx, E)
    assert np.array_equal(off.cpu().numpy(), ref["offsets"])
    assert np.array_equal(row_token.cpu().numpy(), ref["row_token"])
    assert torch.equal(u_perm, u[row_token.long()])


def test_dispatch_zero_tokens():
    shape = S("none", T=0, n_routed=12, top_k=3)
    off = torch.full((13,), -1, dtype=torch.int32, device=DEV)
    ws = M.alloc_workspace(M.moe_dispatch_workspace_size(shape), DEV)
    u = torch.empty((0, shape.H), dtype=torch.bfloat16, device=DEV)
    M.moe_dispatch(shape, None, u, off, None, None, None, ws)
    assert torch.all(off.cpu() == 0)


def test_dispatch_bad_expert_index_is_reported():
    shape = S("bad", T=64, n_routed=8, top_k=2)
    idx = _idx_for(shape, seed=1)
    idx[3, 1] = 99
    u = torch.randn((64, shape.H), device=DEV).to(torch.bfloat16)
    _gpu_dispatch(shape, idx, u)
    st, code = M.moe_device_status()
    assert st == M.MOE_ERR_INVALID_ARG and code & 8
    assert M.moe_device_status() == (M.MOE_OK, 0)   # the word was cleared


# ---------------------------------------------------------------- expert FFN

FFN_SHAPES = [
    S("ffn_swiglu", T=300, H=256, n_routed=8, n_shared=1, top_k=2, inter=128),
    S("ffn_swiglu_tiles", T=1000, H=512, n_routed=4, n_shared=2, top_k=2, inter=192),
    S("ffn_relu", T=200, H=256, n_routed=6, n_shared=1, top_k=2, inter=256, act=W.ACT_RELU),
    S("ffn_decode", T=20, H=384, n_routed=32, n_shared=1, top_k=4, inter=128,
      gate=W.GATE_SIGMOID_BIAS, bias_range=0.1),
    S("ffn_no_shared", T=129, H=256, n_routed=8, n_shared=0, top_k=3, inter=64),
    S("ffn_shared_only", T=77, H=256, n_routed=4, n_shared=2, top_k=0, inter=64),
    S("ffn_long_k", T=100, H=1024, n_routed=16, n_shared=1, top_k=4, inter=1408 // 4 + 32),
    # experts with 257..511 rows (a full tile and a tail), a shared expert
    # whose 2000 rows end in a 208-row tail, an odd number of k-blocks
    S("ffn_wide_tiles", T=2000, H=256, n_routed=8, n_shared=1, top_k=2, inter=128),
    S("ffn_wide_relu", T=700, H=384, n_routed=3, n_shared=1, top_k=1, inter=256,
      act=W.ACT_RELU),
    S("ffn_wide_odd_k", T=900, H=256, n_routed=4, n_shared=1, top_k=1, inter=192),
    dataclasses.replace(W.SHAPES["tiny_f32"], name="ffn_tiny_f32"),
    S("ffn_f32_swiglu", T=150, H=64, n_routed=5, n_shared=1, top_k=2, inter=40, dtype="f32"),
]


@pytest.mark.parametrize("shape", FFN_SHAPES, ids=lambda s: s.name)
def test_expert_ffn(shape):
    inp = W.make_inputs(shape, DEV, seed=11)
    T, k, E, Ks, H = shape.T, shape.top_k, shape.n_routed, shape.n_shared, shape.H
    idx = _idx_for(shape, seed=5, kind="skewed") if k else np.zeros((T, 0), np.int64)
    off, row_token, slot_row, u_perm = _gpu_dispatch(shape, idx, inp.u)
    y_perm = torch.zeros((T * k, H), dtype=shape.torch_dtype, device=DEV)
    y_shared = torch.zeros((Ks, T, H), dtype=shape.torch_dtype, device=DEV)
    ws = M.alloc_workspace(M.moe_expert_ffn_workspace_size(shape), DEV)
    M.moe_expert_ffn(shape, M.weights_struct(inp), inp.u, u_perm, off, y_perm, y_shared, ws)
    torch.cuda.synchronize()
    routed, shared = expert_fns(inp)
    u = np64(inp.u)
    ref = O.dispatch(idx, E)
    tol = TOL[shape.dtype]
    if k:
        yp = np64(y_perm)
        for e in range(E):
            r0, r1 = ref["offsets"][e], ref["offsets"][e + 1]
            if r1 == r0:
                continue
            w1, w3, w2 = routed(e)
            want = O.expert_ffn(u[ref["row_token"][r0:r1]], w1, w2, w3, shape.act)
            assert_close(yp[r0:r1], want, tol, f"routed expert {e}")
    for j in range(Ks):
        w1, w3, w2 = shared(j)
        assert_close(np64(y_shared[j]), O.expert_ffn(u, w1, w2, w3, shape.act), tol,
                     f"shared expert {j}")


# ---------------------------------------------------------------- combine

@pytest.mark.parametrize("dtype,T,H,k,Ks", [("bf16", 333, 512, 6, 2), ("f32", 100, 256, 3, 1),
                                           ("bf16", 50, 7168, 8, 1), ("bf16", 64, 256, 0, 2),
                                           # rows split across warps with a short last
                                           # segment (96, 96, 80 vectors), bf16 and fp32
                                           ("bf16", 1000, 2176, 6, 1), ("f32", 1000, 1088, 4, 1),
                                           ("bf16", 64, 7168, 8, 1)])
def test_combine(dtype, T, H, k, Ks):
    E = max(k, 4)
    shape = S("comb", T=T, H=H, n_routed=E, top_k=k, n_shared=Ks, dtype=dtype)
    g = torch.Generator().manual_seed(T)
    dt = shape.torch_dtype
    u = torch.randn((T, H), generator=g).to(dt)
    y_perm = torch.randn((T * k, H), generator=g).to(dt)
    y_shared = torch.randn((Ks, T, H), generator=g).to(dt)
    w = torch.rand((T, k), generator=g)
    idx = _idx_for(shape, seed=2) if k else np.zeros((T, 0), np.int64)
    slot_row = O.dispatch(idx, E)["slot_row"]
    h = torch.empty((T, H), dtype=dt, device=DEV)
    M.moe_combine(shape, u.to(DEV), y_perm.to(DEV), y_shared.to(DEV), w.to(DEV),
                  torch.from_numpy(slot_row.astype(np.int32)).to(DEV), h)
    yr = np64(y_perm)[slot_row] if k else np.zeros((T, 0, H))
    want = O.combine(np64(u), [np64(y_shared[j]) for j in range(Ks)], yr, np64(w))
    got = np64(h)
    # one rounding to the output type plus fp32 accumulation
    half_ulp = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -23
    mag = np.abs(np64(u)) + sum(np.abs(np64(y_shared[j])) for j in range(Ks)) + \
        (np.abs(yr) * np64(w)[:, :, None]).sum(1)
    assert np.all(np.abs(got - want) <= half_ulp * np.abs(want) + 1e-6 * mag + 1e-30)


def test_combine_zero_gates_is_residual():
    T, H, k = 40, 256, 3
    shape = S("comb0", T=T, H=H, n_routed=6, top_k=k, n_shared=0)
    u = torch.randn((T, H), device=DEV).to(torch.bfloat16)
    y = torch.randn((T * k, H), device=DEV).to(torch.bfloat16)
    slot = torch.arange(T * k, dtype=torch.int32, device=DEV)
    h = torch.empty_like(u)
    M.moe_combine(shape, u, y, None, torch.zeros((T, k), device=DEV), slot, h)
    assert torch.equal(h, u)


# ---------------------------------------------------------------- expert FFN: tile spans

def _idx_with_counts(counts, seed):
    """A top-1 choice in which expert e receives exactly counts[e] tokens, in a
    seeded random token order."""
    idx = np.repeat(np.arange(len(counts)), counts)
    np.random.default_rng(seed).shuffle(idx)
    return idx[:, None]


# Per-expert row counts around the token-tile boundaries of the CTA-pair
# GEMM (256-row tiles, MMA N in steps of 32): empty, one row, one partial
# step, a full tile, a full tile and a one-row tail, tails of every size
# class, several full tiles with and without a tail.
SPAN_COUNTS = [0, 1, 31, 256, 257, 300, 320, 383, 448, 511, 512, 513, 520, 748, 1024, 1025, 1100]


@pytest.mark.parametrize("H,inter,act", [(640, 128, W.ACT_SWIGLU), (1024, 192, W.ACT_SWIGLU),
                                         (384, 256, W.ACT_RELU)])
def test_expert_ffn_tile_spans(H, inter, act):
    """Every routed row and every shared row against the oracle, for expert
    loads on both sides of each token-tile boundary; inter = 192 gives the
    down projection an odd number of k-blocks, the shared expert's rows end in
    a short piece."""
    counts = np.array(SPAN_COUNTS)
    T = int(counts.sum())
    shape = S("ffn_spans", T=T, H=H, n_routed=len(counts), n_shared=1, top_k=1, inter=inter,
              act=act)
    inp = W.make_inputs(shape, DEV, seed=13)
    idx = _idx_with_counts(counts, seed=H)
    off, row_token, slot_row, u_perm = _gpu_dispatch(shape, idx, inp.u)
    E = shape.n_routed
    y_perm = torch.zeros((T, H), dtype=torch.bfloat16, device=DEV)
    y_shared = torch.zeros((1, T, H), dtype=torch.bfloat16, device=DEV)
    ws = M.alloc_workspace(M.moe_expert_ffn_workspace_size(shape), DEV)
    M.moe_expert_ffn(shape, M.weights_struct(inp), inp.u, u_perm, off, y_perm, y_shared, ws)
    st, code = M.moe_device_status()
    assert st == M.MOE_OK, (st, code)
    routed, shared = expert_fns(inp)
    u = np64(inp.u)
    ref = O.dispatch(idx, E)
    assert np.array_equal(np.diff(ref["offsets"]), counts)
    yp = np64(y_perm)
    for e in range(E):
        r0, r1 = ref["offsets"][e], ref["offsets"][e + 1]
        if r1 == r0:
            continue
        w1, w3, w2 = routed(e)
        want = O.expert_ffn(u[ref["row_token"][r0:r1]], w1, w2, w3, act)
        assert_close(yp[r0:r1], want, TOL["bf16"], f"expert {e} ({counts[e]} rows)")
    w1, w3, w2 = shared(0)
    assert_close(np64(y_shared[0]), O.expert_ffn(u, w1, w2, w3, act), TOL["bf16"], "shared")


def test_v3_expert_ffn_whole_experts_full_size():
    """The DeepSeek-V3-shaped layer at full size (K = 7168, 256 routed experts
    with skewed loads from the sigmoid + bias router), moe_expert_ffn in the
    benchmark's launch configuration: every row of the most loaded routed
    expert (two full token tiles and a tail), of one expert with 257..511
    rows (a full tile and a tail on the CTA pair) and of one with at most 256
    rows (one tile), and 512 sampled rows of the shared expert."""
    shape = W.SHAPES["v3_prefill_bf16"]
    inp = W.make_inputs(shape, DEV, seed=0)
    T, E, k, H = shape.T, shape.n_routed, shape.top_k, shape.H
    logits = torch.empty((T, E), dtype=torch.float32, device=DEV)
    M.moe_router_logits(shape, inp.u, inp.centroids, inp.logit_offset, logits)
    idx_t, w_t, _ = gpu_route(shape, logits, inp.select_bias)
    off, row_token, slot_row, u_perm = _gpu_dispatch(shape, idx_t.cpu().numpy(), inp.u)
    y_perm = torch.empty((T * k, H), dtype=torch.bfloat16, device=DEV)
    y_shared = torch.empty((1, T, H), dtype=torch.bfloat16, device=DEV)
    ws = M.alloc_workspace(M.moe_expert_ffn_workspace_size(shape), DEV)
    M.moe_expert_ffn(shape, M.weights_struct(inp), inp.u, u_perm, off, y_perm, y_shared, ws)
    st, code = M.moe_device_status()
    assert st == M.MOE_OK, (st, code)
    offsets = off.cpu().numpy()
    counts = np.diff(offsets)
    heavy = int(np.argmax(counts))
    mid = [e for e in range(E) if 257 <= counts[e] <= 511]
    light = [e for e in range(E) if 0 < counts[e] <= 256]
    assert counts[heavy] > 512 and mid and light, counts
    routed, shared = expert_fns(inp)
    rt = row_token.cpu().numpy()
    for e in (heavy, mid[0], light[0]):
        r0, r1 = offsets[e], offsets[e + 1]
        x = np64(inp.u[torch.from_numpy(rt[r0:r1]).to(DEV).long()])
        w1, w3, w2 = routed(e)
        want = O.expert_ffn(x, w1, w2, w3, shape.act)
        assert_close(np64(y_perm[r0:r1]), want, TOL["bf16"], f"expert {e} ({counts[e]} rows)")
    rows = np.sort(np.random.default_rng(1).choice(T, size=512, replace=False))
    w1, w3, w2 = shared(0)
    want = O.expert_ffn(np64(inp.u)[rows], w1, w2, w3, shape.act)
    assert_close(np64(y_shared[0])[rows], want, TOL["bf16"], "shared expert")
    del inp, y_perm, y_shared, u_perm, ws
    torch.cuda.empty_cache()
