"""The seeded input generator that serves both the kernels and the oracle
(no arithmetic of the method): reproducible draws, the documented shapes,
scales and storage types, and the page-derived layer shapes."""
import math

import numpy as np
import torch

from fine_grained_shared_gemm_b300 import workloads as W


def _small(**kw):
    base = dict(T=64, H=128, n_routed=6, n_shared=2, top_k=2, inter=64)
    base.update(kw)
    return W.MoEShape("gen", **base)


def test_draws_are_reproducible_and_seed_dependent():
    s = _small(gate=W.GATE_SIGMOID_BIAS, bias_range=0.1, logit_offset_std=1.0)
    a, b, c = (W.make_inputs(s, "cpu", seed=x) for x in (0, 0, 1))
    for name in ("u", "centroids", "select_bias", "logit_offset", "w1", "w3", "w2",
                 "sw1", "sw3", "sw2"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
        assert not torch.equal(getattr(a, name), getattr(c, name)), name


def test_shapes_types_and_scales():
    s = _small(T=512, H=256, inter=128)
    inp = W.make_inputs(s, "cpu", seed=0)
    E, Ks, H, I = s.n_routed, s.n_shared, s.H, s.inter
    assert inp.u.shape == (s.T, H) and inp.u.dtype == torch.bfloat16
    assert inp.centroids.shape == (E, H)
    assert inp.w1.shape == (E, I, H) and inp.w3.shape == (E, I, H) and inp.w2.shape == (E, H, I)
    assert inp.sw1.shape == (Ks, I, H) and inp.sw2.shape == (Ks, H, I)
    assert inp.select_bias is None and inp.logit_offset is None      # softmax shape
    # N(0, 1) tokens, N(0, 1/fan_in) weights (loose statistical bounds)
    assert abs(inp.u.float().std().item() - 1.0) < 0.05
    assert abs(inp.w1.float().std().item() * math.sqrt(H) - 1.0) < 0.05
    assert abs(inp.w2.float().std().item() * math.sqrt(I) - 1.0) < 0.05
    relu = W.make_inputs(_small(act=W.ACT_RELU), "cpu", seed=0)
    assert relu.w3 is None and relu.sw3 is None
    f32 = W.make_inputs(_small(dtype="f32"), "cpu", seed=0)
    assert f32.u.dtype == torch.float32


def test_selection_bias_range_and_offsets():
    s = _small(n_routed=64, gate=W.GATE_SIGMOID_BIAS, bias_range=0.1, logit_offset_std=1.0)
    inp = W.make_inputs(s, "cpu", seed=0)
    b = inp.select_bias.numpy()
    assert b.dtype == np.float32 and b.min() >= -0.1 and b.max() <= 0.1
    assert inp.logit_offset.dtype == torch.float32 and inp.logit_offset.shape == (64,)


def test_page_derived_layer_shapes():
    """The 16B row of the model table (64 routed, top-6, 2 shared, hidden
    2048; width 1408) and the V3 row (256 routed, top-8, 1 shared, hidden
    7168, width 2048, sigmoid + bias); the granularity sweep keeps the base
    of 16 experts of width 4096 with 2 active."""
    d = W.SHAPES["dsmoe16b_bf16"]
    assert (d.n_routed, d.top_k, d.n_shared, d.H, d.inter) == (64, 6, 2, 2048, 1408)
    v = W.SHAPES["v3_prefill_bf16"]
    assert (v.n_routed, v.top_k, v.n_shared, v.H, v.inter) == (256, 8, 1, 7168, 2048)
    assert v.gate == W.GATE_SIGMOID_BIAS
    for m in (1, 2, 4, 8, 16):
        s = W.SHAPES[f"sweep_m{m}"]
        assert (s.n_routed, s.top_k, s.inter) == (16 * m, 2 * m, 4096 // m)
        s1 = W.SHAPES[f"sweep_m{m}_shared1"]
        assert (s1.n_routed, s1.n_shared, s1.top_k) == (16 * m - 1, 1, 2 * m - 1)
