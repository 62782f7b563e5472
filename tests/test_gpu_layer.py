"""Whole-layer parity: moe_layer_forward against the oracle.

Small layers are compared on every token.  The page-shaped layers run at
full size in the launch configuration the benchmark times; routing and
dispatch are compared on all T tokens (bit-exact from the kernel's own fp32
logits, near-ties reported), logits and outputs on a seeded sample of tokens
that the oracle evaluates one expert at a time."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from fine_grained_shared_gemm_b300 import moe as M
from fine_grained_shared_gemm_b300 import workloads as W
from parity_helpers import (TOL, assert_close, compare_routing, expert_fns, layer_buffers,
                            np64, oracle_route, route_with_choice)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_layer(shape, inp):
    ws, h = layer_buffers(shape, DEV)
    T, E, k = shape.T, shape.n_routed, shape.top_k
    ro = dict(logits=torch.empty((T, E), dtype=torch.float32, device=DEV),
              topk_idx=torch.empty((T, k), dtype=torch.int32, device=DEV),
              topk_w=torch.empty((T, k), dtype=torch.float32, device=DEV),
              expert_offsets=torch.empty((E + 1,), dtype=torch.int32, device=DEV))
    M.moe_layer_forward(shape, M.weights_struct(inp), inp.u, h, ws, route_out=ro)
    st, code = M.moe_device_status()
    assert st == M.MOE_OK, (st, code)
    return h, ro


def check_layer(shape, inp, h, ro, rows=None):
    """Compare one layer run with the oracle; rows=None compares every token."""
    routed, shared = expert_fns(inp)
    T = shape.T
    gpu_logits = ro["logits"].cpu().numpy()
    # routing, on all tokens, from the kernel's own logits
    ref_route = oracle_route(shape, gpu_logits, inp)
    flipped = compare_routing(shape, ro["topk_idx"], ro["topk_w"], ref_route)
    # dispatch offsets follow from the choice
    d = O.dispatch(ro["topk_idx"].cpu().numpy().astype(np.int64), shape.n_routed)
    assert np.array_equal(ro["expert_offsets"].cpu().numpy(), d["offsets"])
    rows = np.arange(T) if rows is None else np.asarray(rows)
    # logits: oracle's own on the sampled rows
    u = np64(inp.u)
    off = None if inp.logit_offset is None else np64(inp.logit_offset)
    z_ref = O.router_logits(u[rows], np64(inp.centroids), off).astype(np.float64)
    bound = 1e-5 * (np.abs(u[rows]) @ np.abs(np64(inp.centroids)).T) + 1e-6
    assert np.all(np.abs(gpu_logits[rows] - z_ref) <= bound)
    # outputs: the oracle's layer with the kernel's choice on near-tie flips
    choice = ref_route["idx"].copy()
    choice[flipped] = ro["topk_idx"].cpu().numpy()[flipped]
    r = route_with_choice(shape, ref_route, choice)
    want = O.layer_forward(u, r, routed, shared, shape.n_shared, shape.act, rows=rows)
    got = np64(h)[rows]
    err, scale = assert_close(got, want, TOL[shape.dtype], f"layer {shape.name}")
    return dict(err=err, scale=scale, near_ties=int((ref_route["gap"] < 1e-5).sum()),
                flipped=int(flipped.sum()))


SMALL = [
    W.SHAPES["tiny_f32"],
    W.MoEShape("small_softmax", T=500, H=256, n_routed=16, n_shared=2, top_k=4, inter=128),
    W.MoEShape("small_sigmoid", T=333, H=384, n_routed=24, n_shared=1, top_k=6, inter=192,
               gate=W.GATE_SIGMOID_BIAS, bias_range=0.1),
    W.MoEShape("small_decode", T=16, H=512, n_routed=64, n_shared=1, top_k=8, inter=256,
               gate=W.GATE_SIGMOID_BIAS, bias_range=0.1, logit_offset_std=1.0),
    W.MoEShape("small_relu_bf16", T=200, H=256, n_routed=8, n_shared=1, top_k=2, inter=256,
               act=W.ACT_RELU),
    W.MoEShape("classic_top2", T=300, H=256, n_routed=8, n_shared=0, top_k=2, inter=512),
    W.MoEShape("one_token", T=1, H=256, n_routed=8, n_shared=1, top_k=3, inter=64),
    dataclasses.replace(W.SHAPES["tiny_f32"], name="tiny_f32_sigmoid",
                        gate=W.GATE_SIGMOID_BIAS, bias_range=0.1, act=W.ACT_SWIGLU),
    # group-limited routing, V3-style: 64 experts in 8 groups, 4 groups kept
    W.MoEShape("small_groups", T=700, H=256, n_routed=64, n_shared=1, top_k=8, inter=128,
               gate=W.GATE_SIGMOID_BIAS, bias_range=0.1, n_groups=8, topk_groups=4),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_layer_small_all_tokens(shape):
    inp = W.make_inputs(shape, DEV, seed=0)
    h, ro = run_layer(shape, inp)
    check_layer(shape, inp, h, ro)


def test_layer_deterministic_bitwise():
    shape = SMALL[1]
    inp = W.make_inputs(shape, DEV, seed=1)
    h1, _ = run_layer(shape, inp)
    h2, _ = run_layer(shape, inp)
    assert torch.equal(h1, h2)


def test_layer_zero_tokens():
    shape = SMALL[1].with_tokens(0)
    inp = W.make_inputs(shape, DEV, seed=0)
    ws, h = layer_buffers(shape, DEV)
    M.moe_layer_forward(shape, M.weights_struct(inp), inp.u, h, ws)
    assert M.moe_device_status()[0] == M.MOE_OK


def test_layer_host_buffers_match_device_path():
    shape = SMALL[2]
    inp = W.make_inputs(shape, DEV, seed=4)
    h_dev_path, _ = run_layer(shape, inp)
    ws, h = layer_buffers(shape, DEV)
    u_host = inp.u.cpu().pin_memory()
    h_host = torch.empty_like(u_host).pin_memory()
    u_dev = torch.empty_like(inp.u)
    M.moe_layer_forward_host(shape, M.weights_struct(inp), u_host, h_host, u_dev, h, ws)
    torch.cuda.synchronize()
    assert torch.equal(h_host, h_dev_path.cpu())


@pytest.mark.parametrize("n_batches", [1, 2, 5])
def test_layer_host_stream_matches_device_path_batch_by_batch(n_batches):
    """moe_layer_forward_host_stream over distinct host batches: every
    output is bitwise the device-resident forward of its own batch, with
    the copies of neighbouring batches overlapping its layer."""
    shape = SMALL[2]
    inp = W.make_inputs(shape, DEV, seed=8)
    wt = M.weights_struct(inp)
    gen = torch.Generator().manual_seed(9)
    u_hosts = [torch.randn(tuple(inp.u.shape), generator=gen).to(inp.u.dtype).pin_memory()
               for _ in range(n_batches)]
    h_hosts = [torch.zeros_like(u).pin_memory() for u in u_hosts]
    ws, _ = layer_buffers(shape, DEV)
    u_dev = torch.empty((2,) + tuple(inp.u.shape), dtype=inp.u.dtype, device=DEV)
    h_dev = torch.empty_like(u_dev)
    M.moe_layer_forward_host_stream(shape, wt, u_hosts, h_hosts, u_dev, h_dev, ws)
    torch.cuda.synchronize()
    assert M.moe_device_status()[0] == M.MOE_OK
    for b in range(n_batches):
        u = u_hosts[b].to(DEV)
        h = torch.empty_like(u)
        M.moe_layer_forward(shape, wt, u, h, ws)
        torch.cuda.synchronize()
        assert torch.equal(h_hosts[b], h.cpu()), b


def test_layer_host_buffers_pipelined_chunks_match_device_path():
    # enough tokens for the host-buffer entry point to pipeline three chunks
    # (copies on their own streams overlapping the layer on earlier chunks)
    shape = W.MoEShape("host_chunks", T=3 * 4096 + 100, H=256, n_routed=16, n_shared=1,
                       top_k=4, inter=128, gate=W.GATE_SIGMOID_BIAS, bias_range=0.1)
    inp = W.make_inputs(shape, DEV, seed=6)
    h_dev_path, _ = run_layer(shape, inp)
    ws, h = layer_buffers(shape, DEV)
    u_host = inp.u.cpu().pin_memory()
    h_host = torch.zeros_like(u_host).pin_memory()
    u_dev = torch.empty_like(inp.u)
    M.moe_layer_forward_host(shape, M.weights_struct(inp), u_host, h_host, u_dev, h, ws)
    torch.cuda.synchronize()
    assert M.moe_device_status()[0] == M.MOE_OK
    assert torch.equal(h_host, h_dev_path.cpu())


# full-size page-shaped layers: (shape name, sampled tokens; None = every token)
FULL = [("dsmoe16b_bf16", 512), ("v3_prefill_bf16", 512), ("decode_bf16", None),
        ("v3_prefill_e32_bf16", 512), ("sweep_m16_e32_bf16", 512)] + \
    [(f"sweep_m{m}{v}", 512) for v in ("", "_shared1") for m in (1, 2, 4, 8, 16)]


@pytest.mark.parametrize("name,n_sample", FULL, ids=[f[0] for f in FULL])
def test_layer_full_size_sampled(name, n_sample):
    shape = W.SHAPES[name]
    inp = W.make_inputs(shape, DEV, seed=0)
    h, ro = run_layer(shape, inp)
    rows = None if n_sample is None else \
        np.sort(np.random.default_rng(0).choice(shape.T, size=n_sample, replace=False))
    info = check_layer(shape, inp, h, ro, rows=rows)
    print(f"{name}: {info}")
    del inp, h, ro
    torch.cuda.empty_cache()
