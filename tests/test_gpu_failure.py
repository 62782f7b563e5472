"""Failure detection without a GPU fault: a bounded wait that nothing
satisfies expires, sets the device error word, and the context stays usable
(the next layer runs and matches the oracle)."""
import time

import numpy as np
import pytest
import torch

from fine_grained_shared_gemm_b300 import moe as M
from fine_grained_shared_gemm_b300 import workloads as W
from parity_helpers import TOL, assert_close, expert_fns, np64
import oracle.moe_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_bounded_wait_expires_and_context_stays_usable():
    torch.cuda.synchronize()
    assert M.moe_device_status()[0] == M.MOE_OK          # starts clean
    t0 = time.perf_counter()
    M.moe_check_bounded_wait(20000)                       # 20 ms limit
    st, code = M.moe_device_status()
    elapsed = time.perf_counter() - t0
    assert st == M.MOE_ERR_TIMEOUT, (st, code)
    assert code & 2                                       # the MMA-role timeout bit
    assert 0.015 < elapsed < 5.0, elapsed                 # it waited, then gave up
    assert M.moe_device_status()[0] == M.MOE_OK          # reading clears the word
    # the context still works: a small layer matches the oracle
    shape = W.MoEShape("after_timeout", T=300, H=256, n_routed=8, n_shared=1, top_k=2,
                       inter=256)
    inp = W.make_inputs(shape, DEV, seed=0)
    ws = M.alloc_workspace(M.moe_layer_workspace_size(shape), DEV)
    h = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device=DEV)
    logits = torch.empty((shape.T, shape.n_routed), dtype=torch.float32, device=DEV)
    idx = torch.empty((shape.T, shape.top_k), dtype=torch.int32, device=DEV)
    M.moe_layer_forward(shape, M.weights_struct(inp), inp.u, h, ws,
                        route_out={"logits": logits, "topk_idx": idx})
    assert M.moe_device_status()[0] == M.MOE_OK
    # the oracle's layer for the kernel's own choice (routing parity is tested elsewhere)
    choice = idx.cpu().numpy().astype(np.int64)
    r = dict(idx=choice, weights=O.gate_weights(logits.cpu().numpy(), choice, shape.gate)[0])
    routed, shared = expert_fns(inp)
    want = O.layer_forward(np64(inp.u), r, routed, shared, shape.n_shared, shape.act)
    assert_close(np64(h), want, TOL["bf16"], "layer after a timeout")
