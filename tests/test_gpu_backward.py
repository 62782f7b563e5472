"""Layer backward on the GPU against the oracle's backward.

The kernels recompute the forward's routing; the test reads the same
routing from a forward call (same kernels, same inputs) and gives the oracle
that choice, so both sides differentiate the same piecewise-smooth function.
Every gradient tensor is compared element by element at sizes that span
several tiles, ragged tails, experts that nobody chose, the shared-only and
single-token cases; the bar is the layer's bf16 one, max|Δ| ≤ 2e-2 · max|ref|
per tensor (the backward's intermediates are bf16 like the forward's)."""
import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from fine_grained_shared_gemm_b300 import moe as M
from fine_grained_shared_gemm_b300 import workloads as W
from parity_helpers import TOL, assert_close, expert_fns, np64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _shape(name, **kw):
    base = dict(T=200, H=256, n_routed=8, n_shared=1, top_k=2, inter=256, gate=W.GATE_SOFTMAX,
                act=W.ACT_SWIGLU, dtype="bf16")
    base.update(kw)
    return W.MoEShape(name, **base)


SHAPES = [
    _shape("bwd_softmax_swiglu"),
    _shape("bwd_sigmoid_relu_noshared", T=333, n_routed=16, n_shared=0, top_k=4, inter=128,
           gate=W.GATE_SIGMOID_BIAS, act=W.ACT_RELU, bias_range=0.1),
    _shape("bwd_multitile", T=600, H=512, n_routed=6, n_shared=1, top_k=2, inter=384),
    _shape("bwd_narrow_tiles", T=64, H=384, n_routed=32, n_shared=2, top_k=2, inter=128,
           gate=W.GATE_SIGMOID_BIAS, bias_range=0.1),
    _shape("bwd_skewed_empty_experts", T=300, n_routed=12, n_shared=1, top_k=3, inter=128,
           gate=W.GATE_SIGMOID_BIAS, bias_range=0.1, logit_offset_std=3.0),
    _shape("bwd_shared_only", T=130, n_routed=4, n_shared=2, top_k=0, inter=128),
    _shape("bwd_one_token", T=1, n_routed=8, n_shared=1, top_k=2, inter=128),
    # group-limited routing (V3 style): 32 experts in 8 groups, 3 groups kept
    _shape("bwd_groups", T=400, n_routed=32, n_shared=1, top_k=4, inter=128,
           gate=W.GATE_SIGMOID_BIAS, bias_range=0.1, n_groups=8, topk_groups=3),
    # H above 4096: the derivative epilogue on four warps; I = 384 leaves the
    # second CTA of the last pair tile no features
    _shape("bwd_wide_h_four_warps", T=90, H=4224, n_routed=6, n_shared=1, top_k=2, inter=384),
]


def grads_buffers(shape):
    E, Ks, H, I = shape.n_routed, shape.n_shared, shape.H, shape.inter
    sw = shape.act == W.ACT_SWIGLU
    f = lambda *s: torch.full(s, float("nan"), dtype=torch.float32, device=DEV)
    g = dict(d_centroids=f(E, H), dw1=f(E, I, H), dw3=f(E, I, H) if sw else None, dw2=f(E, H, I),
             dsw1=f(Ks, I, H) if Ks else None, dsw3=f(Ks, I, H) if Ks and sw else None,
             dsw2=f(Ks, H, I) if Ks else None)
    return g


def run_backward(shape, inp, dh, saved=None):
    g = grads_buffers(shape)
    du = torch.full((shape.T, shape.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = M.alloc_workspace(M.moe_layer_backward_workspace_size(shape), DEV)
    M.moe_layer_backward(shape, M.weights_struct(inp), inp.u, dh, du,
                         M.weight_grads(g["d_centroids"], g["dw1"], g["dw3"], g["dw2"],
                                        g["dsw1"], g["dsw3"], g["dsw2"]), ws, saved=saved)
    st, code = M.moe_device_status()
    assert st == M.MOE_OK, (st, code)
    return du, g


def forward_routing(shape, inp):
    T, E, k = shape.T, shape.n_routed, shape.top_k
    ws = M.alloc_workspace(M.moe_layer_workspace_size(shape), DEV)
    h = torch.empty((T, shape.H), dtype=torch.bfloat16, device=DEV)
    ro = dict(logits=torch.empty((T, E), dtype=torch.float32, device=DEV),
              topk_idx=torch.empty((T, k), dtype=torch.int32, device=DEV))
    M.moe_layer_forward(shape, M.weights_struct(inp), inp.u, h, ws, route_out=ro)
    return ro["logits"].cpu().numpy(), ro["topk_idx"].cpu().numpy().astype(np.int64)


def oracle_backward(shape, inp, dh, z, idx):
    routed, shared = expert_fns(inp)
    return O.layer_backward(np64(inp.u), np64(dh), np64(inp.centroids), z, idx, shape.gate,
                            routed, shared, shape.n_routed, shape.n_shared, shape.act)


def forward_train(shape, inp):
    """moe_layer_forward_train: h and the saved buffer."""
    ws = M.alloc_workspace(M.moe_layer_workspace_size(shape), DEV)
    saved = M.alloc_workspace(M.moe_layer_saved_size(shape), DEV)
    h = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device=DEV)
    M.moe_layer_forward_train(shape, M.weights_struct(inp), inp.u, h, saved, ws)
    return h, saved


@pytest.mark.parametrize("mode", ["recompute", "saved"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_layer_backward_matches_oracle(shape, mode):
    inp = W.make_inputs(shape, DEV, seed=0)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(1)
    dh = torch.randn((shape.T, shape.H), generator=gen, device=DEV).to(torch.bfloat16)
    saved = forward_train(shape, inp)[1] if mode == "saved" else None
    du, g = run_backward(shape, inp, dh, saved)
    torch.cuda.synchronize()
    z, idx = forward_routing(shape, inp)
    ref = oracle_backward(shape, inp, dh, z, idx)
    tol = TOL["bf16"]
    assert_close(np64(du), ref["du"], tol, "du")
    if shape.top_k > 0:
        assert_close(np64(g["d_centroids"]), ref["d_centroids"], tol, "d_centroids")
    else:
        assert not g["d_centroids"].any()
    for key in ("dw1", "dw3", "dw2", "dsw1", "dsw3", "dsw2"):
        if g[key] is None:
            assert ref[key] is None or ref[key].size == 0, key
            continue
        got = np64(g[key])
        assert np.isfinite(got).all(), key
        if ref[key] is None or not np.abs(ref[key]).any():
            assert not got.any(), key        # nobody chose any expert: exact zeros
        else:
            assert_close(got, ref[key], tol, key)
    # experts nobody chose get exact zeros
    counts = np.bincount(idx.reshape(-1), minlength=shape.n_routed) if shape.top_k else \
        np.zeros(shape.n_routed, np.int64)
    for e in np.nonzero(counts == 0)[0]:
        for key in ("dw1", "dw3", "dw2"):
            if g[key] is not None:
                assert not g[key][e].any(), (key, e)


def test_skewed_case_has_empty_experts():
    """The skewed shape above really exercises empty experts (zero-length
    contractions in the weight-gradient GEMMs)."""
    shape = [s for s in SHAPES if s.name == "bwd_skewed_empty_experts"][0]
    inp = W.make_inputs(shape, DEV, seed=0)
    _, idx = forward_routing(shape, inp)
    counts = np.bincount(idx.reshape(-1), minlength=shape.n_routed)
    assert (counts == 0).any(), counts


def test_layer_backward_is_deterministic():
    shape = SHAPES[2]
    inp = W.make_inputs(shape, DEV, seed=0)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(2)
    dh = torch.randn((shape.T, shape.H), generator=gen, device=DEV).to(torch.bfloat16)
    du1, g1 = run_backward(shape, inp, dh)
    du2, g2 = run_backward(shape, inp, dh)
    torch.cuda.synchronize()
    assert torch.equal(du1, du2)
    for key in g1:
        if g1[key] is not None:
            assert torch.equal(g1[key], g2[key]), key


def test_backward_rejects_unsupported_shapes():
    bad = _shape("bwd_f32", dtype="f32", inter=128)
    assert M.moe_layer_backward_workspace_size(bad) == 0
    odd = _shape("bwd_odd_inter", inter=192)
    assert M.moe_layer_backward_workspace_size(odd) == 0


# Full-size page-shaped layers in the configuration the benchmark times:
# (shape name, sampled tokens for du, sampled routed experts for dW; the most
# loaded expert is always among them).
FULL = [("dsmoe16b_bf16", 64, 8), ("v3_prefill_bf16", 64, 8)]


@pytest.mark.parametrize("name,n_tok,n_exp", FULL, ids=[f[0] for f in FULL])
def test_layer_backward_full_size_sampled(name, n_tok, n_exp):
    """du on sampled tokens (each token's gradient depends only on that
    token), the weight gradients of sampled routed experts (over all the rows
    that chose them) and of the first shared expert (over all tokens).  The
    centroid gradient sums dz over every token, which needs every expert's
    output for every token: it is checked on the small layers and on the
    mid-size layer below."""
    shape = W.SHAPES[name]
    inp = W.make_inputs(shape, DEV, seed=0)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(1)
    dh = torch.randn((shape.T, shape.H), generator=gen, device=DEV).to(torch.bfloat16)
    du, g = run_backward(shape, inp, dh)
    torch.cuda.synchronize()
    z, idx = forward_routing(shape, inp)
    routed, shared = expert_fns(inp)
    rng = np.random.default_rng(0)
    u, dh64, cents = np64(inp.u), np64(dh), np64(inp.centroids)
    tol = TOL["bf16"]
    # du on sampled tokens
    rows = np.sort(rng.choice(shape.T, size=n_tok, replace=False))
    ref = O.layer_backward(u[rows], dh64[rows], cents, z[rows], idx[rows], shape.gate, routed,
                           shared, shape.n_routed, shape.n_shared, shape.act,
                           experts=np.unique(idx[rows]))
    assert_close(np64(du)[rows], ref["du"], tol, f"{name} du")
    # weight gradients of sampled routed experts: every row that chose them
    gw, _ = O.gate_weights(z, idx, shape.gate)
    counts = np.bincount(idx.reshape(-1), minlength=shape.n_routed)
    heavy = int(np.argmax(counts))
    others = np.setdiff1d(np.nonzero(counts)[0], [heavy])
    for e in [heavy] + list(rng.choice(others, size=n_exp - 1, replace=False)):
        tt, ss = np.nonzero(idx == e)
        w1, w3, w2 = routed(int(e))
        _, dw1, dw3, dw2 = O.expert_ffn_backward(u[tt], w1, w2, w3, shape.act,
                                                 gw[tt, ss][:, None] * dh64[tt])
        assert_close(np64(g["dw1"][e]), dw1, tol, f"{name} dw1[{e}]")
        assert_close(np64(g["dw2"][e]), dw2, tol, f"{name} dw2[{e}]")
        if dw3 is not None:
            assert_close(np64(g["dw3"][e]), dw3, tol, f"{name} dw3[{e}]")
    # the first shared expert: every token
    w1, w3, w2 = shared(0)
    _, dw1, dw3, dw2 = O.expert_ffn_backward(u, w1, w2, w3, shape.act, dh64)
    assert_close(np64(g["dsw1"][0]), dw1, tol, f"{name} dsw1[0]")
    assert_close(np64(g["dsw2"][0]), dw2, tol, f"{name} dsw2[0]")
    if dw3 is not None:
        assert_close(np64(g["dsw3"][0]), dw3, tol, f"{name} dsw3[0]")
    del inp, du, g
    torch.cuda.empty_cache()


@pytest.mark.parametrize("shape", SHAPES[:3], ids=lambda s: s.name)
def test_training_forward_matches_forward(shape):
    """The training forward gives the forward's h bit for bit."""
    inp = W.make_inputs(shape, DEV, seed=3)
    h_train, _ = forward_train(shape, inp)
    ws = M.alloc_workspace(M.moe_layer_workspace_size(shape), DEV)
    h = torch.empty_like(h_train)
    M.moe_layer_forward(shape, M.weights_struct(inp), inp.u, h, ws)
    torch.cuda.synchronize()
    assert M.moe_device_status()[0] == M.MOE_OK
    assert torch.equal(h, h_train)


@pytest.mark.parametrize("shape", [SHAPES[2], SHAPES[3]], ids=lambda s: s.name)
def test_training_step_replays_from_a_cuda_graph(shape):
    """moe_layer_forward_train and moe_layer_backward make no host
    synchronisation or allocation: both capture into one CUDA graph, and its
    replays give the eager calls' h, du and weight gradients bit for bit."""
    inp = W.make_inputs(shape, DEV, seed=7)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(8)
    dh = torch.randn((shape.T, shape.H), generator=gen, device=DEV).to(torch.bfloat16)
    h_ref, saved_ref = forward_train(shape, inp)
    du_ref, g_ref = run_backward(shape, inp, dh, saved_ref)
    # fresh buffers, captured once
    wt = M.weights_struct(inp)
    ws_f = M.alloc_workspace(M.moe_layer_workspace_size(shape), DEV)
    ws_b = M.alloc_workspace(M.moe_layer_backward_workspace_size(shape), DEV)
    saved = M.alloc_workspace(M.moe_layer_saved_size(shape), DEV)
    h = torch.empty_like(h_ref)
    du = torch.empty_like(du_ref)
    g = grads_buffers(shape)
    grads = M.weight_grads(g["d_centroids"], g["dw1"], g["dw3"], g["dw2"], g["dsw1"], g["dsw3"],
                           g["dsw2"])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        M.moe_layer_forward_train(shape, wt, inp.u, h, saved, ws_f)
        M.moe_layer_backward(shape, wt, inp.u, dh, du, grads, ws_b, saved=saved)
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        assert M.moe_device_status()[0] == M.MOE_OK
        assert torch.equal(h, h_ref)
        assert torch.equal(du, du_ref)
        for key, t in g.items():
            if t is not None:
                assert torch.equal(t, g_ref[key]), key
        h.zero_()
        du.zero_()


def test_autograd_layer_matches_oracle():
    """The torch.autograd wrapper: gradients of sum(h * dh) through a PyTorch
    model equal the oracle's backward for the kernels' own choice."""
    from fine_grained_shared_gemm_b300.autograd import MoELayer
    shape = _shape("bwd_autograd", T=256, n_routed=8, n_shared=1, top_k=2, inter=128,
                   gate=W.GATE_SIGMOID_BIAS)
    layer = MoELayer(shape, DEV, seed=5)
    with torch.no_grad():
        layer.select_bias.uniform_(-0.1, 0.1)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(6)
    u = torch.randn((shape.T, shape.H), generator=gen, device=DEV).to(torch.bfloat16)
    u.requires_grad_(True)
    dh = torch.randn((shape.T, shape.H), generator=gen, device=DEV).to(torch.bfloat16)
    h = layer(u)
    (h.float() * dh.float()).sum().backward()
    torch.cuda.synchronize()
    assert M.moe_device_status()[0] == M.MOE_OK
    # the kernels' choice, from a plain forward of the same layer
    T, E, k = shape.T, shape.n_routed, shape.top_k
    ws = M.alloc_workspace(M.moe_layer_workspace_size(shape), DEV)
    ro = dict(logits=torch.empty((T, E), dtype=torch.float32, device=DEV),
              topk_idx=torch.empty((T, k), dtype=torch.int32, device=DEV))
    h2 = torch.empty_like(h)
    from fine_grained_shared_gemm_b300.autograd import _weights
    wt = _weights(layer.centroids, layer.w1, layer.w3, layer.w2, layer.sw1, layer.sw3,
                  layer.sw2, None, layer.select_bias)
    M.moe_layer_forward(shape, wt, u.detach(), h2, ws, route_out=ro)
    assert torch.equal(h.detach(), h2)
    f = lambda t: np64(t.detach())
    routed = lambda e: (f(layer.w1[e]), f(layer.w3[e]), f(layer.w2[e]))
    shared = lambda j: (f(layer.sw1[j]), f(layer.sw3[j]), f(layer.sw2[j]))
    ref = O.layer_backward(f(u), f(dh), f(layer.centroids), ro["logits"].cpu().numpy(),
                           ro["topk_idx"].cpu().numpy().astype(np.int64), shape.gate, routed,
                           shared, E, shape.n_shared, shape.act)
    tol = TOL["bf16"]
    assert_close(f(u.grad), ref["du"], tol, "du")
    for name, key in (("centroids", "d_centroids"), ("w1", "dw1"), ("w3", "dw3"), ("w2", "dw2"),
                      ("sw1", "dsw1"), ("sw3", "dsw3"), ("sw2", "dsw2")):
        grad = getattr(layer, name).grad
        assert grad is not None and grad.dtype == torch.bfloat16, name
        # the parameter's bf16 gradient against the oracle (one more rounding)
        assert_close(f(grad), ref[key], tol, name)


def test_layer_backward_mid_size_every_gradient():
    """A mid-size layer (2048 tokens, H = 2048, 64 routed experts with several
    token tiles each, two shared experts) where the oracle can evaluate every
    token: du, the centroid gradient (a sum of dz over all 2048 tokens) and
    every weight gradient, element by element."""
    shape = _shape("bwd_mid", T=2048, H=2048, n_routed=64, n_shared=2, top_k=6, inter=512)
    inp = W.make_inputs(shape, DEV, seed=0)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(1)
    dh = torch.randn((shape.T, shape.H), generator=gen, device=DEV).to(torch.bfloat16)
    du, g = run_backward(shape, inp, dh)
    torch.cuda.synchronize()
    z, idx = forward_routing(shape, inp)
    ref = oracle_backward(shape, inp, dh, z, idx)
    tol = TOL["bf16"]
    assert_close(np64(du), ref["du"], tol, "du")
    assert_close(np64(g["d_centroids"]), ref["d_centroids"], tol, "d_centroids")
    for key in ("dw1", "dw3", "dw2", "dsw1", "dsw3", "dsw2"):
        assert_close(np64(g[key]), ref[key], tol, key)
