"""The aux-loss-free bias controller (page "MoE 的分水岭", ch. 7 §7.4) on the
GPU against the oracle: bit-exact updates, and a closed loop that evens out a
skewed router when routing, dispatch and the update all run in the kernels."""
import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from fine_grained_shared_gemm_b300 import moe as M
from fine_grained_shared_gemm_b300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("T,E,k", [(6, 4, 2), (1000, 64, 6), (333, 257, 8), (5, 16, 3)])
def test_bias_update_bit_exact(T, E, k):
    rng = np.random.default_rng(T + E)
    # loads that sum to T*k, several exactly at the mean when it is an integer
    loads = rng.multinomial(T * k, np.ones(E) / E)
    if (T * k) % E == 0:
        loads[:] = (T * k) // E
        for i in range(0, E - 1, 3):   # move rows between neighbours, keep the sum
            d = min(loads[i], 1 + i % 2)
            loads[i] -= d
            loads[i + 1] += d
    offsets = np.concatenate([[0], np.cumsum(loads)]).astype(np.int32)
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    gamma = 1e-3
    shape = W.MoEShape("balance", T=T, H=128, n_routed=E, n_shared=0, top_k=k, inter=64)
    b_dev = torch.from_numpy(bias.copy()).to(DEV)
    loads_dev = torch.full((E,), -1, dtype=torch.int32, device=DEV)
    M.moe_update_select_bias(shape, torch.from_numpy(offsets).to(DEV), b_dev, gamma, loads_dev)
    torch.cuda.synchronize()
    want = O.update_select_bias(loads, bias, gamma, T * k)
    assert np.array_equal(b_dev.cpu().numpy(), want)
    assert np.array_equal(loads_dev.cpu().numpy(), loads.astype(np.int32))


def test_bias_controller_closed_loop_on_gpu():
    """Routing, dispatch and the bias update run in the kernels for many steps;
    each step's update equals the oracle's for the kernels' own loads, and the
    most loaded expert ends within 1.12x of the mean."""
    T, H, E, k = 4096, 256, 32, 4
    gen = torch.Generator(device=DEV)
    gen.manual_seed(0)
    u = torch.randn((T, H), generator=gen, device=DEV).to(torch.bfloat16)
    scale = torch.linspace(0.02, 0.4, E, device=DEV)[:, None] / H ** 0.5 * 4
    cents = (torch.randn((E, H), generator=gen, device=DEV) * scale).to(torch.bfloat16)
    shape = W.MoEShape("loop", T=T, H=H, n_routed=E, n_shared=0, top_k=k, inter=64,
                       gate=W.GATE_SIGMOID_BIAS)
    logits = torch.empty((T, E), dtype=torch.float32, device=DEV)
    M.moe_router_logits(shape, u, cents, None, logits)
    bias = torch.zeros(E, dtype=torch.float32, device=DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    off = torch.empty((E + 1,), dtype=torch.int32, device=DEV)
    row_token = torch.empty((T * k,), dtype=torch.int32, device=DEV)
    slot_row = torch.empty((T * k,), dtype=torch.int32, device=DEV)
    u_perm = torch.empty((T * k, H), dtype=torch.bfloat16, device=DEV)
    ws = M.alloc_workspace(M.moe_dispatch_workspace_size(shape), DEV)
    loads = torch.empty((E,), dtype=torch.int32, device=DEV)
    imbalance = []
    for _ in range(300):
        M.moe_route(shape, logits, bias, idx, w)
        M.moe_dispatch(shape, idx, u, off, row_token, slot_row, u_perm, ws)
        before = bias.cpu().numpy()
        M.moe_update_select_bias(shape, off, bias, 2e-3, loads)
        torch.cuda.synchronize()
        got_loads = loads.cpu().numpy()
        assert got_loads.sum() == T * k
        assert np.array_equal(bias.cpu().numpy(),
                              O.update_select_bias(got_loads, before, 2e-3, T * k))
        imbalance.append(got_loads.max() * E / (T * k))
    assert M.moe_device_status()[0] == M.MOE_OK
    assert imbalance[0] > 1.6, imbalance[0]
    assert max(imbalance[-20:]) < 1.12, imbalance[-20:]


@pytest.mark.parametrize("gate", [W.GATE_SOFTMAX, W.GATE_SIGMOID_BIAS])
@pytest.mark.parametrize("T,E,k", [(1, 4, 2), (255, 64, 6), (1000, 257, 8), (4097, 16, 3)])
def test_balance_stats_against_oracle(gate, T, E, k):
    """f_i and P_i of the expert-level balance loss (page "19-deepseek-moe",
    load-balance section) from the kernels' own logits, routing and dispatch:
    f bit-exact (an exact integer ratio rounded once), P within 1e-5 of its
    largest entry (fp32 scores and sums of at most 256 terms; the oracle sums
    float64 scores)."""
    gen = torch.Generator(device=DEV)
    gen.manual_seed(T * 7 + E)
    H = 128
    u = torch.randn((T, H), generator=gen, device=DEV).to(torch.bfloat16)
    cents = (torch.randn((E, H), generator=gen, device=DEV) / H ** 0.5 * 3).to(torch.bfloat16)
    shape = W.MoEShape("stats", T=T, H=H, n_routed=E, n_shared=0, top_k=k, inter=64, gate=gate)
    logits = torch.empty((T, E), dtype=torch.float32, device=DEV)
    M.moe_router_logits(shape, u, cents, None, logits)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    M.moe_route(shape, logits, None, idx, w)
    off = torch.empty((E + 1,), dtype=torch.int32, device=DEV)
    row_token = torch.empty((T * k,), dtype=torch.int32, device=DEV)
    slot_row = torch.empty((T * k,), dtype=torch.int32, device=DEV)
    u_perm = torch.empty((T * k, H), dtype=torch.bfloat16, device=DEV)
    M.moe_dispatch(shape, idx, u, off, row_token, slot_row, u_perm,
                   M.alloc_workspace(M.moe_dispatch_workspace_size(shape), DEV))
    f = torch.full((E,), float("nan"), dtype=torch.float32, device=DEV)
    p = torch.full((E,), float("nan"), dtype=torch.float32, device=DEV)
    ws = M.alloc_workspace(M.moe_balance_stats_workspace_size(shape), DEV)
    M.moe_balance_stats(shape, logits, off, f, p, ws)
    torch.cuda.synchronize()
    assert M.moe_device_status()[0] == M.MOE_OK
    want_f, want_p = O.balance_stats(logits.cpu().numpy(), idx.cpu().numpy(), E, k,
                                     O.SOFTMAX if gate == W.GATE_SOFTMAX else O.SIGMOID_BIAS)
    assert np.array_equal(f.cpu().numpy(), want_f)
    got_p = p.cpu().numpy().astype(np.float64)
    assert np.abs(got_p - want_p).max() <= 1e-5 * want_p.max(), np.abs(got_p - want_p).max()
    assert abs(got_p.sum() - 1.0) < 1e-4
    # a second call gives the same bits (fixed-order sums)
    p2 = torch.empty_like(p)
    M.moe_balance_stats(shape, logits, off, f, p2, ws)
    torch.cuda.synchronize()
    assert torch.equal(p, p2)
