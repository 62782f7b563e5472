"""Expert parallelism over two gloo ranks on the CPU (no GPU).

Each rank routes and dispatches its own tokens (the oracle does the local
arithmetic here), then the product's exchange code moves the per-expert
counts and the token rows to the rank that holds their expert and back
(page "02 · 细粒度 MoE：从 Mixtral 到 DeepSeekMoE", §3.2: routed experts
spread over devices, rows exchanged all-to-all, shared experts replicated).
Checked: the counts and the received rows bit for bit against the layout
derived from every rank's routing, and the combined output of each rank
against the oracle's layer over all tokens in one process."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle.moe_oracle as O
from fine_grained_shared_gemm_b300 import expert_parallel as EP
from fine_grained_shared_gemm_b300 import workloads as W

WORLD = 2
E, K, KS, H, I = 8, 3, 1, 64, 32
T_RANK = [37, 50]          # tokens per rank (ragged)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer_inputs():
    shape = W.MoEShape("ep_gloo", T=sum(T_RANK), H=H, n_routed=E, n_shared=KS, top_k=K,
                       inter=I, gate=W.GATE_SIGMOID_BIAS, act=W.ACT_SWIGLU, dtype="f32",
                       bias_range=0.1)
    return shape, W.make_inputs(shape, "cpu", seed=0)


def _f64(t):
    return t.detach().to(torch.float64).numpy()


def _worker(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        shape, inp = _layer_inputs()
        el = E // WORLD
        t0 = sum(T_RANK[:rank])
        u = _f64(inp.u)[t0:t0 + T_RANK[rank]]
        bias = inp.select_bias.numpy()
        # local routing and dispatch (the oracle's arithmetic on this rank's tokens)
        z = O.router_logits(u, _f64(inp.centroids))
        r = O.route(z, shape.gate, K, bias)
        d = O.dispatch(r["idx"], E)
        u_perm = u[d["row_token"]]
        send_counts = np.diff(d["offsets"])
        # the product's exchange: counts, split sizes, rows
        recv_counts = EP.exchange_counts(send_counts, WORLD, "cpu")
        send_splits = EP.rank_splits(send_counts, WORLD)
        recv_splits = EP.rank_splits(recv_counts, WORLD)
        x_recv = torch.empty((int(recv_counts.sum()), H), dtype=torch.float64)
        EP.exchange_rows(x_recv, torch.from_numpy(u_perm), recv_splits, send_splits)
        # local experts of this rank on the received rows, regrouped expert-major
        # and back (the order moe_ep_regroup implements on the GPU)
        cm = recv_counts.reshape(WORLD, el)
        src_off = np.concatenate([[0], np.cumsum(cm.reshape(-1))])
        y_recv = np.empty_like(x_recv.numpy())
        for e in range(el):
            blocks = [(src_off[s * el + e], cm[s, e]) for s in range(WORLD)]
            rows = np.concatenate([np.arange(a, a + n) for a, n in blocks])
            ge = rank * el + e
            w = (_f64(inp.w1[ge]), _f64(inp.w3[ge]), _f64(inp.w2[ge]))
            if rows.size:
                y_recv[rows] = O.expert_ffn(x_recv.numpy()[rows], w[0], w[2], w[1], shape.act)
        y_perm = torch.empty((u_perm.shape[0], H), dtype=torch.float64)
        EP.exchange_rows(y_perm, torch.from_numpy(y_recv), send_splits, recv_splits)
        # shared experts on the local tokens, combine in the local dispatch order
        y_sh = [O.expert_ffn(u, _f64(inp.sw1[j]), _f64(inp.sw2[j]), _f64(inp.sw3[j]), shape.act)
                for j in range(KS)]
        h = O.combine(u, y_sh, y_perm.numpy()[d["slot_row"]], r["weights"])
        # everything every rank needs to check the layout
        gathered = [None] * WORLD
        dist.all_gather_object(gathered, dict(idx=r["idx"], u_perm=u_perm,
                                              offsets=d["offsets"]))
        out.put((rank, recv_counts, x_recv.numpy(), h, gathered))
    finally:
        dist.destroy_process_group()


def test_two_rank_expert_parallel_exchange_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = mp.spawn(_worker, args=(_free_port(), q), nprocs=WORLD, join=False)
    # read the results before joining: a child cannot exit while its queued
    # data is unread
    res = sorted([q.get(timeout=120) for _ in range(WORLD)], key=lambda x: x[0])
    procs.join()
    shape, inp = _layer_inputs()
    el = E // WORLD
    gathered = res[0][4]
    for rank, recv_counts, x_recv, h, _ in res:
        # counts: source s sends its rows for expert rank·E_loc + e
        want_counts = np.concatenate([np.diff(gathered[s]["offsets"])[rank * el:(rank + 1) * el]
                                      for s in range(WORLD)])
        assert np.array_equal(recv_counts, want_counts)
        # rows, bit for bit: source-major, then expert, then the source's dispatch order
        want_rows = np.concatenate([
            gathered[s]["u_perm"][gathered[s]["offsets"][rank * el]:
                                  gathered[s]["offsets"][(rank + 1) * el]]
            for s in range(WORLD)])
        assert np.array_equal(x_recv, want_rows)
    # combined outputs against the oracle's layer over all tokens at once
    u = _f64(inp.u)
    z = O.router_logits(u, _f64(inp.centroids))
    r = O.route(z, shape.gate, K, inp.select_bias.numpy())
    routed = lambda e: (_f64(inp.w1[e]), _f64(inp.w3[e]), _f64(inp.w2[e]))
    shared = lambda j: (_f64(inp.sw1[j]), _f64(inp.sw3[j]), _f64(inp.sw2[j]))
    want = O.layer_forward(u, r, routed, shared, KS, shape.act)
    got = np.concatenate([x[3] for x in res])
    assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want))
    # the routing really spreads rows over both ranks' experts
    assert all(x[1].sum() > 0 for x in res)


def test_rank_splits():
    assert EP.rank_splits(np.array([1, 2, 0, 5, 3, 0]), 3) == [3, 5, 3]
    assert EP.rank_splits(np.zeros(4, np.int64), 2) == [0, 0]
