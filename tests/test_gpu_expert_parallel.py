"""Expert-parallel layer forward on the GPU: D ranks held in one process on
one device (the all-to-all exchanges become device-to-device copies), every
step of each rank in the CUDA library.  Checked per rank: the regrouped rows
and offsets bit for bit against the layout derived from all ranks' routing,
and the output against the oracle's layer on that rank's tokens (routing
from the kernels' own fp32 logits, near-ties reported as in the layer tests).
The multi-process path over NCCL runs the same per-rank steps; its exchange
code is covered on the CPU by the gloo test."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from fine_grained_shared_gemm_b300 import expert_parallel as EP
from fine_grained_shared_gemm_b300 import moe as M
from fine_grained_shared_gemm_b300 import workloads as W
from parity_helpers import (TOL, assert_close, compare_routing, expert_fns, np64, oracle_route,
                            route_with_choice)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CASES = [
    # (name, layer shape over all ranks' tokens, tokens per rank)
    ("softmax_d4", W.MoEShape("ep_softmax", T=0, H=512, n_routed=64, n_shared=2, top_k=6,
                              inter=256), [300, 257, 700, 1]),
    ("sigmoid_d2", W.MoEShape("ep_sigmoid", T=0, H=1024, n_routed=32, n_shared=1, top_k=4,
                              inter=512, gate=W.GATE_SIGMOID_BIAS, bias_range=0.1),
     [1200, 900]),
    ("d8_no_shared", W.MoEShape("ep_noshared", T=0, H=256, n_routed=64, n_shared=0, top_k=8,
                                inter=128, gate=W.GATE_SIGMOID_BIAS, bias_range=0.1,
                                logit_offset_std=1.0), [64] * 8),
    ("d1", W.MoEShape("ep_d1", T=0, H=256, n_routed=16, n_shared=1, top_k=4, inter=128),
     [333]),
]


@pytest.mark.parametrize("name,shape,t_rank", CASES, ids=[c[0] for c in CASES])
def test_expert_parallel_virtual_ranks(name, shape, t_rank):
    D = len(t_rank)
    full = dataclasses.replace(shape, T=sum(t_rank))
    inp = W.make_inputs(full, DEV, seed=0)
    starts = np.concatenate([[0], np.cumsum(t_rank)])
    ranks, us = [], []
    for d in range(D):
        rs = dataclasses.replace(shape, T=t_rank[d])
        ranks.append(EP.ExpertParallelRank(rs, EP.shard_weights(inp, d, D), d, D, DEV))
        us.append(inp.u[starts[d]:starts[d + 1]].contiguous())
    hs = EP.forward_virtual(ranks, us)
    st, code = M.moe_device_status()
    assert st == M.MOE_OK, (st, code)
    el = shape.n_routed // D
    # layout: rank d received, source-major, the rows every source dispatched to
    # its experts, and its expert-major offsets follow
    offs = [r.off.cpu().numpy() for r in ranks]
    u_perms = [r.u_perm for r in ranks]
    for d, r in enumerate(ranks):
        want = torch.cat([u_perms[s][int(offs[s][d * el]):int(offs[s][(d + 1) * el])]
                          for s in range(D)])
        assert torch.equal(r.x_recv, want)
        counts = np.stack([np.diff(offs[s])[d * el:(d + 1) * el] for s in range(D)])
        assert np.array_equal(r.recv_counts.reshape(D, el), counts)
    # outputs against the oracle, rank by rank
    routed, shared = expert_fns(inp)
    worst = 0.0
    for d, r in enumerate(ranks):
        rs = r.shape
        ref_route = oracle_route(rs, r.logits.cpu().numpy(), inp)
        flipped = compare_routing(rs, r.idx, r.w, ref_route)
        choice = ref_route["idx"].copy()
        choice[flipped] = r.idx.cpu().numpy()[flipped]
        rr = route_with_choice(rs, ref_route, choice)
        want = O.layer_forward(np64(us[d]), rr, routed, shared, rs.n_shared, rs.act)
        err, scale = assert_close(np64(hs[d]), want, TOL["bf16"], f"{name} rank {d}")
        worst = max(worst, err / max(scale, 1e-30))
    print(f"{name}: worst max|Δ|/max|ref| = {worst:.2e}")


def test_expert_parallel_matches_single_device_layer():
    """The expert-parallel path and moe_layer_forward on the same tokens use the
    same kernels and summation orders: their outputs agree to the bf16 bar
    (and are usually identical)."""
    name, shape, t_rank = CASES[1]
    D = len(t_rank)
    full = dataclasses.replace(shape, T=sum(t_rank))
    inp = W.make_inputs(full, DEV, seed=2)
    starts = np.concatenate([[0], np.cumsum(t_rank)])
    ranks = [EP.ExpertParallelRank(dataclasses.replace(shape, T=t_rank[d]),
                                   EP.shard_weights(inp, d, D), d, D, DEV) for d in range(D)]
    us = [inp.u[starts[d]:starts[d + 1]].contiguous() for d in range(D)]
    hs = EP.forward_virtual(ranks, us)
    for d in range(D):
        rs = dataclasses.replace(shape, T=t_rank[d])
        ws = M.alloc_workspace(M.moe_layer_workspace_size(rs), DEV)
        h = torch.empty_like(us[d])
        M.moe_layer_forward(rs, M.weights_struct(inp), us[d], h, ws)
        torch.cuda.synchronize()
        assert_close(np64(hs[d]), np64(h), TOL["bf16"], f"rank {d}")


def test_ep_regroup_round_trip_and_offsets():
    """moe_ep_regroup both ways: source-major -> expert-major -> source-major is
    the identity, and the expert-major order and offsets follow the counts."""
    D, el, H = 3, 5, 256
    shape = W.MoEShape("regroup", T=1, H=H, n_routed=el, n_shared=0, top_k=0, inter=64)
    g = torch.Generator().manual_seed(0)
    counts = torch.randint(0, 40, (D, el), generator=g)
    counts[1, 2] = 0
    n = int(counts.sum())
    x = torch.randn((n, H), generator=g).to(torch.bfloat16).to(DEV)
    c_dev = counts.reshape(-1).to(torch.int32).to(DEV)
    y = torch.empty_like(x)
    off = torch.full((el + 1,), -1, dtype=torch.int32, device=DEV)
    M.moe_ep_regroup(shape, D, c_dev, n, x, y, off, to_expert_major=True)
    back = torch.empty_like(x)
    M.moe_ep_regroup(shape, D, c_dev, n, y, back, None, to_expert_major=False)
    torch.cuda.synchronize()
    assert torch.equal(back, x)
    cm = counts.numpy()
    src_off = np.concatenate([[0], np.cumsum(cm.reshape(-1))]).reshape(-1)
    want = torch.cat([x[int(src_off[s * el + e]):int(src_off[s * el + e]) + int(cm[s, e])]
                      for e in range(el) for s in range(D)])
    assert torch.equal(y, want)
    assert np.array_equal(off.cpu().numpy(),
                          np.concatenate([[0], np.cumsum(cm.sum(axis=0))]))
