"""Layer shapes and seeded synthetic inputs for the DeepSeekMoE layer forward.

This module holds no arithmetic of the method itself: it only names the layer
shapes that the source pages describe and draws seeded random tensors of those
shapes.  Both the CUDA path (through the binding) and the CPU oracle consume
what it produces; neither side's arithmetic lives here.

Sources for the shapes (page titles as printed on the pages):

* "02 · 细粒度 MoE：从 Mixtral 到 DeepSeekMoE" (llm-infra-atlas), §2.1 gives
  the segmentation rule (N experts of width M become mN experts of width M/m,
  mK active), §3.1 the shared-expert isolation (Ks always-on experts, routed
  top-k lowered to mK-Ks), §4's table the DeepSeekMoE-16B row (64 routed,
  top-6, 2 shared, hidden 2048) and the DeepSeek-V3 row (256 routed, top-8,
  1 shared, hidden 7168, sigmoid) and the Kimi K2 row (384 routed, top-8,
  1 shared, hidden 7168).
* "MoE 的分水岭——DeepSeek 配方与 2026 年的主流形态" (ibossgateway, ch. 7),
  §7.4: the per-expert selection bias b_i that only affects the choice.

Value distributions: tokens u ~ N(0, 1); every weight matrix ~ N(0, 1/fan_in)
where fan_in is the contracted dimension (H for W1, W3 and the routing
centroids, the expert width I for W2); V3-style selection bias b_i ~ U(-0.1,
0.1); the decode shape additionally adds a per-expert logit offset o_i ~ N(0, 1)
to the router logits so that expert loads are uneven.  All draws come from one
torch generator seeded with ``seed`` in the fixed order: u, centroids,
selection bias, logit offsets, then per expert (shared experts first, then
routed) W1, W3, W2.  The generator is the one of the device the tensors are
made on, so values made on a GPU differ from values made on the CPU; the
oracle is always fed the exact values the kernels see.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import torch

GATE_SOFTMAX = "softmax"
GATE_SIGMOID_BIAS = "sigmoid_bias"
ACT_RELU = "relu"
ACT_SWIGLU = "swiglu"


@dataclass(frozen=True)
class MoEShape:
    """One MoE layer's shape.

    T tokens of hidden size H; ``n_routed`` routed experts of which ``top_k``
    are chosen per token; ``n_shared`` always-on shared experts; every expert
    (shared or routed) has intermediate width ``inter``.  ``gate`` is the
    scoring rule, ``act`` the expert FFN form, ``dtype`` the storage type of
    tokens, weights and output ("f32" or "bf16").
    """

    name: str
    T: int
    H: int
    n_routed: int
    n_shared: int
    top_k: int
    inter: int
    gate: str = GATE_SOFTMAX
    act: str = ACT_SWIGLU
    dtype: str = "bf16"
    bias_range: float = 0.0          # b_i ~ U(-bias_range, bias_range); 0 = no bias
    logit_offset_std: float = 0.0    # o_i ~ N(0, std^2); 0 = no offset
    # group-limited routing: n_groups groups of n_routed / n_groups experts,
    # topk_groups of them kept per token; 0 = no limit
    n_groups: int = 0
    topk_groups: int = 0
    # Segmentation provenance (None where the shape is quoted directly):
    # N base FFNs of width M, granularity m, K active base FFNs.
    seg: Optional[tuple] = field(default=None)
    description: str = ""

    def with_tokens(self, T: int) -> "MoEShape":
        return replace(self, T=T)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def n_mats(self) -> int:
        return 3 if self.act == ACT_SWIGLU else 2


def _sweep(m: int, shared: bool) -> MoEShape:
    # Base: N=16 SwiGLU FFNs of width M=4096, K=2 active; granularity m.
    N, M, K = 16, 4096, 2
    ks = 1 if shared else 0
    return MoEShape(
        name=f"sweep_m{m}{'_shared1' if shared else ''}",
        T=16384, H=2048, n_routed=m * N - ks, n_shared=ks, top_k=m * K - ks,
        inter=M // m, gate=GATE_SOFTMAX, act=ACT_SWIGLU, dtype="bf16",
        seg=(N, M, m, K),
        description=(f"granularity sweep m={m}: {m * N} experts of width {M // m}"
                     + (", 1 shared + top-(mK-1)" if shared else ", top-mK")),
    )


SHAPES = {
    s.name: s
    for s in [
        MoEShape(
            name="tiny_f32", T=256, H=256, n_routed=14, n_shared=2, top_k=6,
            inter=64, gate=GATE_SOFTMAX, act=ACT_RELU, dtype="f32",
            seg=(4, 256, 4, 2),
            description="tiny fp32 layer: N=4 FFNs of M=256 split m=4 into 16 "
                        "experts of width 64, 2 shared + 14 routed, top-6, ReLU"),
        MoEShape(
            name="dsmoe16b_bf16", T=16384, H=2048, n_routed=64, n_shared=2,
            top_k=6, inter=1408, gate=GATE_SOFTMAX, act=ACT_SWIGLU, dtype="bf16",
            description="DeepSeekMoE-16B-shaped layer: 2 shared + 64 routed "
                        "SwiGLU experts of width 1408, top-6 softmax"),
        *[_sweep(m, sh) for sh in (False, True) for m in (1, 2, 4, 8, 16)],
        MoEShape(
            name="v3_prefill_bf16", T=8192, H=7168, n_routed=256, n_shared=1,
            top_k=8, inter=2048, gate=GATE_SIGMOID_BIAS, act=ACT_SWIGLU,
            dtype="bf16", bias_range=0.1,
            description="DeepSeek-V3-shaped prefill layer: 1 shared + 256 routed "
                        "SwiGLU experts of width 2048, top-8 sigmoid + bias"),
        # Smaller layers with the same per-expert GEMM shapes as two of the
        # layers above (same H, width and rows per expert, fewer experts), for
        # hardware-counter captures that must stay a few GB on the device.
        MoEShape(
            name="v3_prefill_e32_bf16", T=1024, H=7168, n_routed=32, n_shared=1,
            top_k=8, inter=2048, gate=GATE_SIGMOID_BIAS, act=ACT_SWIGLU,
            dtype="bf16", bias_range=0.1,
            description="V3-shaped prefill layer cut to 32 routed experts and 1024 "
                        "tokens: 256 rows per expert as in the full layer"),
        MoEShape(
            name="dsmoe16b_e16_bf16", T=4096, H=2048, n_routed=16, n_shared=2,
            top_k=6, inter=1408, gate=GATE_SOFTMAX, act=ACT_SWIGLU, dtype="bf16",
            description="DeepSeekMoE-16B-shaped layer cut to 16 routed experts and "
                        "4096 tokens: 1536 rows per routed expert as in the full layer"),
        MoEShape(
            name="sweep_m16_e32_bf16", T=16384, H=2048, n_routed=32, n_shared=0,
            top_k=4, inter=256, gate=GATE_SOFTMAX, act=ACT_SWIGLU, dtype="bf16",
            description="granularity m=16 expert shape (width 256, 2048 rows per "
                        "expert) with 32 experts"),
        MoEShape(
            name="decode_e48_bf16", T=8, H=7168, n_routed=48, n_shared=1, top_k=8,
            inter=2048, gate=GATE_SIGMOID_BIAS, act=ACT_SWIGLU, dtype="bf16",
            bias_range=0.1, logit_offset_std=1.0,
            description="decode-shaped layer cut to 48 routed experts and 8 tokens: "
                        "about 1.3 routed rows per expert as in the full decode layer"),
        MoEShape(
            name="decode_bf16", T=64, H=7168, n_routed=384, n_shared=1, top_k=8,
            inter=2048, gate=GATE_SIGMOID_BIAS, act=ACT_SWIGLU, dtype="bf16",
            bias_range=0.1, logit_offset_std=1.0,
            description="decode-shaped layer: 64 tokens, 1 shared + 384 routed "
                        "SwiGLU experts of width 2048, top-8 sigmoid + bias, "
                        "skewed logits"),
    ]
}


@dataclass
class MoEInputs:
    """Seeded tensors for one layer (all on one device).

    Weight layout (row-major, the contracted dimension contiguous):
      centroids [E, H];  w1, w3 [E, I, H];  w2 [E, H, I];
      sw1, sw3 [Ks, I, H];  sw2 [Ks, H, I]   (w3/sw3 are None for ReLU).
    select_bias and logit_offset are fp32 [E] or None.
    """

    shape: MoEShape
    u: torch.Tensor
    centroids: torch.Tensor
    select_bias: Optional[torch.Tensor]
    logit_offset: Optional[torch.Tensor]
    w1: torch.Tensor
    w3: Optional[torch.Tensor]
    w2: torch.Tensor
    sw1: torch.Tensor
    sw3: Optional[torch.Tensor]
    sw2: torch.Tensor


def _normal(gen, shape, std, dtype, device):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def make_inputs(shape: MoEShape, device="cpu", seed: int = 0) -> MoEInputs:
    """Draw a layer's inputs and weights in the documented order."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    dt = shape.torch_dtype
    T, H, E, Ks, I = shape.T, shape.H, shape.n_routed, shape.n_shared, shape.inter
    swiglu = shape.act == ACT_SWIGLU

    u = _normal(gen, (T, H), 1.0, dt, device)
    centroids = _normal(gen, (E, H), H ** -0.5, dt, device)
    select_bias = None
    if shape.bias_range > 0:
        r = torch.rand((E,), generator=gen, device=device, dtype=torch.float32)
        select_bias = (r * 2.0 - 1.0) * shape.bias_range
    logit_offset = None
    if shape.logit_offset_std > 0:
        logit_offset = _normal(gen, (E,), shape.logit_offset_std, torch.float32, device)

    def stack(n):
        w1 = torch.empty((n, I, H), dtype=dt, device=device)
        w3 = torch.empty((n, I, H), dtype=dt, device=device) if swiglu else None
        w2 = torch.empty((n, H, I), dtype=dt, device=device)
        return w1, w3, w2

    sw1, sw3, sw2 = stack(Ks)
    w1, w3, w2 = stack(E)
    for (a1, a3, a2), n in (((sw1, sw3, sw2), Ks), ((w1, w3, w2), E)):
        for e in range(n):
            a1[e] = _normal(gen, (I, H), H ** -0.5, dt, device)
            if swiglu:
                a3[e] = _normal(gen, (I, H), H ** -0.5, dt, device)
            a2[e] = _normal(gen, (H, I), I ** -0.5, dt, device)
    return MoEInputs(shape, u, centroids, select_bias, logit_offset,
                     w1, w3, w2, sw1, sw3, sw2)


def make_token_inputs(shape: MoEShape, device="cpu", seed: int = 0) -> dict:
    """The routing inputs of a layer only (u, centroids, selection bias, logit
    offsets), equal to those of :func:`make_inputs` with the same seed: they
    are the first draws of the documented order.  For timing the kernels that
    never read expert weights without allocating them."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    T, H, E = shape.T, shape.H, shape.n_routed
    u = _normal(gen, (T, H), 1.0, shape.torch_dtype, device)
    centroids = _normal(gen, (E, H), H ** -0.5, shape.torch_dtype, device)
    select_bias = None
    if shape.bias_range > 0:
        r = torch.rand((E,), generator=gen, device=device, dtype=torch.float32)
        select_bias = (r * 2.0 - 1.0) * shape.bias_range
    logit_offset = None
    if shape.logit_offset_std > 0:
        logit_offset = _normal(gen, (E,), shape.logit_offset_std, torch.float32, device)
    return dict(u=u, centroids=centroids, select_bias=select_bias, logit_offset=logit_offset)


def random_logits(T: int, E: int, device="cpu", seed: int = 0,
                  kind: str = "normal") -> torch.Tensor:
    """fp32 router logits for routing-only tests.

    kind = "normal": N(0, 1); "ties": small integers so that many exact ties
    occur; "skewed": N(0, 1) plus a per-expert N(0, 3^2) offset so that loads
    are very uneven and some experts get no token.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    if kind == "normal":
        return torch.randn((T, E), generator=gen, device=device)
    if kind == "ties":
        return torch.randint(-2, 3, (T, E), generator=gen, device=device).float()
    if kind == "skewed":
        z = torch.randn((T, E), generator=gen, device=device)
        off = torch.randn((E,), generator=gen, device=device) * 3.0
        return z + off
    raise ValueError(kind)
