"""moe_dispatch_static: dispatch for callers that cannot allocate device memory.

Some callers cannot hand the library scratch memory: a serving runtime whose
allocator has reserved all of the GPU's memory up front, or a latency-critical
path that must not call cudaMalloc because it can synchronise the device.
For them the library offers moe_dispatch_static, which keeps its scratch in a
fixed array of its own.  This test checks, through the C ABI, that it gives
exactly what moe_dispatch gives (dispatch is index work, so the comparison is
bit-exact) on two calls in a row, the second reusing the array the first left
behind, and that a shape beyond the array's capacity is refused before any
launch.  The file name makes pytest collect it after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from fine_grained_shared_gemm_b300 import moe as M
from fine_grained_shared_gemm_b300 import workloads as W

DEV = "cuda:0"


def _outputs(shape, dev):
    T, k, E, H = shape.T, shape.top_k, shape.n_routed, shape.H
    return (torch.full((E + 1,), -1, dtype=torch.int32, device=dev),
            torch.full((T * k,), -1, dtype=torch.int32, device=dev),
            torch.full((T * k,), -1, dtype=torch.int32, device=dev),
            torch.zeros((T * k, H), dtype=torch.bfloat16, device=dev))


@pytest.mark.gpu
def test_static_scratch_dispatch_matches_workspace_dispatch():
    # two different layers in a row: the second call finds the first call's
    # leftovers in the shared array
    for shape, seed in ((W.MoEShape("noalloc_a", T=5000, H=256, n_routed=64, n_shared=1,
                                    top_k=6, inter=128), 1),
                        (W.MoEShape("noalloc_b", T=777, H=512, n_routed=256, n_shared=1,
                                    top_k=8, inter=128), 2)):
        z = W.random_logits(shape.T, shape.n_routed, seed=seed, kind="skewed").numpy()
        idx = torch.from_numpy(O.route(z, W.GATE_SOFTMAX, shape.top_k)["idx"]
                               .astype(np.int32)).to(DEV)
        u = torch.randn((shape.T, shape.H), device=DEV).to(torch.bfloat16)

        ref = _outputs(shape, DEV)
        ws = M.alloc_workspace(M.moe_dispatch_workspace_size(shape), DEV)
        M.moe_dispatch(shape, idx, u, *ref, ws)

        got = _outputs(shape, DEV)
        M.moe_dispatch_static(shape, idx, u, *got)
        torch.cuda.synchronize()
        assert M.moe_device_status() == (M.MOE_OK, 0)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


@pytest.mark.gpu
def test_static_scratch_dispatch_refuses_oversize_shapes():
    # ceil(T / 256) * n_routed above the array's 131072 entries.  Every buffer
    # is real and large enough for the shape, so that if the size check ever
    # ran after the launches the call would still stay inside its buffers and
    # this test would fail on the status, not fault the GPU.
    shape = W.MoEShape("noalloc_big", T=256 * 129, H=256, n_routed=1024, n_shared=0,
                       top_k=8, inter=128)
    idx = torch.zeros((shape.T, shape.top_k), dtype=torch.int32, device=DEV)
    idx += torch.arange(shape.top_k, dtype=torch.int32, device=DEV)
    u = torch.zeros((shape.T, shape.H), dtype=torch.bfloat16, device=DEV)
    out = _outputs(shape, DEV)
    st = M.lib().moe_dispatch_static(ctypes.byref(M.shape_struct(shape)), M._ptr(idx),
                                     M._ptr(u), *[M._ptr(t) for t in out], None)
    torch.cuda.synchronize()
    assert st == M.MOE_ERR_UNSUPPORTED
    assert M.moe_device_status() == (M.MOE_OK, 0)
    assert bool((out[0] == -1).all())      # nothing was launched
