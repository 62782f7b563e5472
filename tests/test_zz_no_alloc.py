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
    # ceil(T / 256) * n_routed above the array's 131072 entries
    big = M.moe_shape(T=256 * 129, H=256, n_routed=1024, n_shared=0, top_k=8, inter=128,
                      gate=0, act=1, dtype=1)
    st = M.lib().moe_dispatch_static(ctypes.byref(big), 256, 256, 256, 256, 256, 256, None)
    assert st == M.MOE_ERR_UNSUPPORTED
