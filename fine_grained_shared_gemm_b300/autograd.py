"""PyTorch autograd wrapper of the layer's training calls (argument marshalling
only): the forward is ``moe_layer_forward_train``, the backward is
``moe_layer_backward`` on the tensors that call kept.  Both run in the CUDA
library; nothing here computes.

Gradients flow to the tokens u, the centroids and every expert weight.  The
selection bias only changes which experts are chosen and the logit offset is
treated as a constant, so neither receives one (as the C ABI documents).  The
library returns weight gradients in fp32; autograd casts them to the
parameters' dtype.
"""
from __future__ import annotations

import math
from typing import Optional

import torch

from . import moe as M
from .workloads import ACT_SWIGLU, MoEShape


def _weights(centroids, w1, w3, w2, sw1, sw3, sw2, logit_offset, select_bias):
    p = M._ptr
    return M.moe_weights(p(centroids), p(logit_offset), p(select_bias), p(w1), p(w3), p(w2),
                         p(sw1), p(sw3), p(sw2))


class MoELayerFunction(torch.autograd.Function):
    """h = layer(u) with the chosen experts recorded at the forward."""

    @staticmethod
    def forward(ctx, shape: MoEShape, u, centroids, w1, w3, w2, sw1, sw3, sw2,
                logit_offset: Optional[torch.Tensor], select_bias: Optional[torch.Tensor]):
        dev = u.device
        wt = _weights(centroids, w1, w3, w2, sw1, sw3, sw2, logit_offset, select_bias)
        ws = M.alloc_workspace(M.moe_layer_workspace_size(shape), dev)
        saved = M.alloc_workspace(M.moe_layer_saved_size(shape), dev)
        h = torch.empty_like(u)
        M.moe_layer_forward_train(shape, wt, u, h, saved, ws)
        ctx.shape = shape
        ctx.saved_buffer = saved
        ctx.save_for_backward(u, centroids, w1, w3, w2, sw1, sw3, sw2, logit_offset, select_bias)
        return h

    @staticmethod
    def backward(ctx, dh):
        u, centroids, w1, w3, w2, sw1, sw3, sw2, logit_offset, select_bias = ctx.saved_tensors
        s = ctx.shape
        dev = u.device
        f32 = lambda t: None if t is None else torch.empty(t.shape, dtype=torch.float32,
                                                           device=dev)
        g = [f32(centroids), f32(w1), f32(w3), f32(w2), f32(sw1), f32(sw3), f32(sw2)]
        du = torch.empty_like(u)
        wt = _weights(centroids, w1, w3, w2, sw1, sw3, sw2, logit_offset, select_bias)
        bws = M.alloc_workspace(M.moe_layer_backward_workspace_size(s), dev)
        M.moe_layer_backward(s, wt, u, dh.to(u.dtype).contiguous(), du, M.weight_grads(*g), bws,
                             saved=ctx.saved_buffer)
        return (None, du, g[0], g[1], g[2], g[3], g[4], g[5], g[6], None, None)


class MoELayer(torch.nn.Module):
    """The layer as a module: bf16 parameters centroids [E, H], w1, w3 [E, I, H],
    w2 [E, H, I] and the shared experts' sw1, sw3 [Ks, I, H], sw2 [Ks, H, I]
    (w3 / sw3 absent for ReLU), N(0, 1/fan_in) initialised; the selection bias
    (sigmoid gate) is a buffer, updated by :meth:`update_select_bias`.  The
    forward takes u [T, H] with T = shape.T."""

    def __init__(self, shape: MoEShape, device="cuda:0", seed: int = 0):
        super().__init__()
        self.shape = shape
        E, Ks, H, I = shape.n_routed, shape.n_shared, shape.H, shape.inter
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)
        sw = shape.act == ACT_SWIGLU

        def param(*dims, fan_in):
            if dims[0] == 0:
                return None
            t = torch.randn(dims, generator=gen, device=device) / math.sqrt(fan_in)
            return torch.nn.Parameter(t.to(torch.bfloat16))

        self.centroids = param(E, H, fan_in=H)
        self.w1 = param(E, I, H, fan_in=H)
        self.w3 = param(E, I, H, fan_in=H) if sw else None
        self.w2 = param(E, H, I, fan_in=I)
        self.sw1 = param(Ks, I, H, fan_in=H)
        self.sw3 = param(Ks, I, H, fan_in=H) if sw else None
        self.sw2 = param(Ks, H, I, fan_in=I)
        self.register_buffer("select_bias", torch.zeros(E, device=device))

    def forward(self, u: torch.Tensor) -> torch.Tensor:
        bias = self.select_bias if self.shape.gate == "sigmoid_bias" else None
        return MoELayerFunction.apply(self.shape, u, self.centroids, self.w1, self.w3, self.w2,
                                      self.sw1, self.sw3, self.sw2, None, bias)

    @torch.no_grad()
    def update_select_bias(self, expert_offsets: torch.Tensor, gamma: float, loads=None):
        """One step of the aux-loss-free bias controller (moe_update_select_bias)."""
        M.moe_update_select_bias(self.shape, expert_offsets, self.select_bias, gamma, loads)
