"""The layer shards by batch with no exchange: two gloo ranks on the CPU.

Each rank evaluates its half of a batch with the oracle; gathered, the halves
equal the whole batch evaluated at once (tokens are independent).  The
timing reduction bench.py uses under torchrun returns the slowest rank's time.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle.moe_oracle as O
from fine_grained_shared_gemm_b300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer(shape, inp, rows):
    f64 = lambda t: t.to(torch.float64).numpy()
    u = f64(inp.u)[rows]
    z = O.router_logits(u, f64(inp.centroids))
    r = O.route(z, shape.gate, shape.top_k)
    routed = lambda e: (f64(inp.w1[e]), None, f64(inp.w2[e]))
    shared = lambda j: (f64(inp.sw1[j]), None, f64(inp.sw2[j]))
    return O.layer_forward(u, r, routed, shared, shape.n_shared, shape.act)


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(1.5 + rank, torch.device("cpu"))
        shape = W.SHAPES["tiny_f32"].with_tokens(64)
        inp = W.make_inputs(shape, "cpu", seed=0)
        rows = np.arange(rank, shape.T, world)          # this rank's shard
        h = torch.from_numpy(_layer(shape, inp, rows))
        parts = [torch.empty_like(h) for _ in range(world)]
        dist.all_gather(parts, h)
        if rank == 0:
            full = _layer(shape, inp, np.arange(shape.T))
            merged = np.empty_like(full)
            for r in range(world):
                merged[np.arange(r, shape.T, world)] = parts[r].numpy()
            out.put((slowest, float(np.max(np.abs(merged - full)))))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    mp.spawn(_worker, args=(2, port, q), nprocs=2, join=True)
    slowest, err = q.get(timeout=60)
    assert slowest == 2.5
    assert err < 1e-12   # float64 BLAS may block a shard differently from the batch


def _rate_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 2 + r seconds for its 1000 tokens
        value, slowest = bench.whole_job_rate(1000, 2.0 + rank, world, torch.device("cpu"))
        out.put((rank, value, slowest))
    finally:
        dist.destroy_process_group()


def test_whole_job_rate_counts_every_rank_over_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    mp.spawn(_rate_worker, args=(2, _free_port(), q), nprocs=2, join=True)
    got = sorted(q.get(timeout=60) for _ in range(2))
    for rank, value, slowest in got:
        assert slowest == 3.0                 # the slowest rank's time on every rank
        assert value == 2000 / 3.0            # both ranks' tokens over that time
