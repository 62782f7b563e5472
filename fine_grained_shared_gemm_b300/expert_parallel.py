"""Expert-parallel layer forward over D ranks (argument marshalling and
collectives only: every step on the data path runs in the CUDA library, the
exchanges are torch.distributed all-to-all calls, NCCL on GPUs).

Page "02 · 细粒度 MoE：从 Mixtral 到 DeepSeekMoE" (llm-infra-atlas), §3.2:
the routed experts are spread over the devices and token rows travel to
them and back by all-to-all; the shared experts are replicated on every
device, see every local token and need no exchange.  Here rank d of D holds
the routed experts [d·E_loc, (d+1)·E_loc), E_loc = E / D, every shared
expert and every routing centroid, and a batch of its own tokens.  One step:

  1. router logits, route and dispatch on the local tokens (the full E-way
     routing; dispatch sorts rows by expert, so the rows for each rank are
     one contiguous block, in rank order);
  2. the shared experts start on a side stream (they overlap steps 3-6);
  3. all-to-all of the per-expert row counts (E_loc per destination), then
     of the rows themselves;
  4. the received rows (source-major) are regrouped expert-major;
  5. the local routed experts run on them (moe_expert_ffn_rows);
  6. the outputs are regrouped source-major and sent back by the reverse
     all-to-all, landing in the local dispatch order;
  7. combine with the local gate weights and the shared outputs.

The row counts cross to the host once per step (the all-to-all needs the
split sizes there).  ``forward`` runs one rank per process under
torch.distributed; ``forward_virtual`` runs D ranks in one process on one
device, with the exchanges done as device-to-device copies, so that the
whole path can be exercised with a single GPU.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np
import torch

from . import moe as M
from .workloads import ACT_SWIGLU, MoEInputs, MoEShape


@dataclasses.dataclass
class EPWeights:
    """One rank's parameters: all routing tensors, its E_loc routed experts,
    every shared expert (device tensors, layouts as in include/moe.h)."""

    centroids: torch.Tensor
    select_bias: Optional[torch.Tensor]
    logit_offset: Optional[torch.Tensor]
    w1: torch.Tensor
    w3: Optional[torch.Tensor]
    w2: torch.Tensor
    sw1: torch.Tensor
    sw3: Optional[torch.Tensor]
    sw2: torch.Tensor


def shard_weights(inp: MoEInputs, rank: int, world: int) -> EPWeights:
    """Rank `rank`'s share of a layer's parameters (contiguous expert block)."""
    E = inp.shape.n_routed
    if E % world:
        raise ValueError(f"{E} routed experts do not split evenly over {world} ranks")
    el = E // world
    sl = slice(rank * el, (rank + 1) * el)
    pick = lambda t: None if t is None else t[sl].contiguous()
    return EPWeights(inp.centroids, inp.select_bias, inp.logit_offset, pick(inp.w1),
                     pick(inp.w3), pick(inp.w2), inp.sw1, inp.sw3, inp.sw2)


def rank_splits(counts: np.ndarray, world: int) -> List[int]:
    """Rows per rank from per-expert counts laid out rank-major ([world · E_loc])."""
    c = np.asarray(counts, dtype=np.int64).reshape(world, -1)
    return [int(x) for x in c.sum(axis=1)]


def exchange_counts(send_counts: np.ndarray, world: int, device, group=None) -> np.ndarray:
    """All-to-all of per-expert row counts: send_counts [E] (rank-major: the
    E_loc experts of rank 0 first) -> recv_counts [world · E_loc], the counts
    each source rank sends to this rank's experts, source-major."""
    import torch.distributed as dist
    t = torch.from_numpy(np.asarray(send_counts, dtype=np.int32)).to(device)
    out = torch.empty_like(t)
    dist.all_to_all_single(out, t, group=group)
    return out.cpu().numpy().astype(np.int64)


def exchange_rows(recv: torch.Tensor, send: torch.Tensor, recv_splits: Sequence[int],
                  send_splits: Sequence[int], group=None):
    """All-to-all of token rows with per-rank split sizes (rows of send go to
    the ranks in order; rows from every source land in recv in rank order)."""
    import torch.distributed as dist
    dist.all_to_all_single(recv, send, list(recv_splits), list(send_splits), group=group)


class ExpertParallelRank:
    """The per-rank state and steps of one expert-parallel layer forward.

    ``shape`` is the layer's (T = this rank's tokens, n_routed = all E)."""

    def __init__(self, shape: MoEShape, weights: EPWeights, rank: int, world: int, device):
        if shape.n_routed % world:
            raise ValueError("routed experts must split evenly over the ranks")
        if shape.dtype != "bf16" and shape.dtype != "f32":
            raise ValueError(shape.dtype)
        self.shape, self.rank, self.world = shape, rank, world
        self.device = torch.device(device)
        self.el = shape.n_routed // world
        base = dict(n_routed=self.el, top_k=0, n_groups=0, topk_groups=0)
        self.routed_shape = dataclasses.replace(shape, n_shared=0, **base)
        self.shared_shape = dataclasses.replace(shape, **base)
        w = weights
        self.weights = w
        self.wt_local = M.moe_weights(None, None, None, M._ptr(w.w1), M._ptr(w.w3), M._ptr(w.w2),
                                      M._ptr(w.sw1) if w.sw1.numel() else None,
                                      M._ptr(w.sw3) if w.sw3 is not None and w.sw3.numel()
                                      else None,
                                      M._ptr(w.sw2) if w.sw2.numel() else None)
        self.side = torch.cuda.Stream(self.device)
        self.zero_offsets = torch.zeros(self.el + 1, dtype=torch.int32, device=self.device)
        self._keep = None

    # ---- step 1-2: local routing, dispatch, shared experts on the side stream
    def begin(self, u: torch.Tensor) -> np.ndarray:
        s, dev = self.shape, self.device
        T, E, k, H = u.shape[0], s.n_routed, s.top_k, s.H
        if T != s.T:
            raise ValueError(f"rank batch has {T} tokens, shape says {s.T}")
        self.u = u
        self.logits = torch.empty((T, E), dtype=torch.float32, device=dev)
        self.idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.w = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.off = torch.empty((E + 1,), dtype=torch.int32, device=dev)
        self.row_token = torch.empty((T * k,), dtype=torch.int32, device=dev)
        self.slot_row = torch.empty((T * k,), dtype=torch.int32, device=dev)
        self.u_perm = torch.empty((T * k, H), dtype=u.dtype, device=dev)
        ws_d = M.alloc_workspace(M.moe_dispatch_workspace_size(s), dev)
        M.moe_router_logits(s, u, self.weights.centroids, self.weights.logit_offset, self.logits)
        M.moe_route(s, self.logits, self.weights.select_bias, self.idx, self.w)
        M.moe_dispatch(s, self.idx, u, self.off, self.row_token, self.slot_row, self.u_perm, ws_d)
        # the shared experts need no exchange: they run while the rows travel
        self.y_shared = torch.empty((s.n_shared, T, H), dtype=u.dtype, device=dev)
        if s.n_shared:
            self.side.wait_stream(torch.cuda.current_stream(dev))
            ws_s = M.alloc_workspace(
                M.moe_expert_ffn_rows_workspace_size(self.shared_shape, 0), dev)
            with torch.cuda.stream(self.side):
                M.moe_expert_ffn_rows(self.shared_shape, self.wt_local, 0, u, None,
                                      self.zero_offsets, None, self.y_shared, ws_s)
            self._keep = (ws_s, u)
        offsets = self.off.cpu().numpy().astype(np.int64)   # host: split sizes
        return np.diff(offsets)

    # ---- step 3: split sizes from the exchanged counts, receive buffer
    def receive_counts(self, recv_counts: np.ndarray):
        """recv_counts [world · E_loc] source-major.  Returns (send rows,
        send splits, receive buffer, receive splits) for the row exchange."""
        self.send_splits = rank_splits(self.send_counts_of(), self.world)
        self.recv_counts = np.asarray(recv_counts, dtype=np.int64)
        self.recv_splits = rank_splits(self.recv_counts, self.world)
        self.n_recv = int(self.recv_counts.sum())
        self.x_recv = torch.empty((self.n_recv, self.shape.H), dtype=self.u.dtype,
                                  device=self.device)
        return self.u_perm, self.send_splits, self.x_recv, self.recv_splits

    def send_counts_of(self) -> np.ndarray:
        return np.diff(self.off.cpu().numpy().astype(np.int64))

    # ---- steps 4-6: regroup, local experts, regroup back
    def experts(self):
        """Returns (output rows to send back, their splits, the buffer they
        land in on this rank, its splits) for the reverse exchange."""
        dev, R, H = self.device, self.n_recv, self.shape.H
        counts = torch.from_numpy(self.recv_counts.astype(np.int32)).to(dev)
        x_loc = torch.empty_like(self.x_recv)
        loc_off = torch.empty((self.el + 1,), dtype=torch.int32, device=dev)
        M.moe_ep_regroup(self.routed_shape, self.world, counts, R, self.x_recv, x_loc, loc_off,
                         to_expert_major=True)
        y_loc = torch.empty_like(x_loc)
        ws_r = M.alloc_workspace(M.moe_expert_ffn_rows_workspace_size(self.routed_shape, R), dev)
        M.moe_expert_ffn_rows(self.routed_shape, self.wt_local, R, self.u, x_loc, loc_off, y_loc,
                              None, ws_r)
        y_send = torch.empty_like(y_loc)
        M.moe_ep_regroup(self.routed_shape, self.world, counts, R, y_loc, y_send, None,
                         to_expert_major=False)
        self.y_perm = torch.empty_like(self.u_perm)
        return y_send, self.recv_splits, self.y_perm, self.send_splits

    # ---- step 7: combine
    def finish(self) -> torch.Tensor:
        s = self.shape
        torch.cuda.current_stream(self.device).wait_stream(self.side)
        self._keep = None   # the side stream's buffers are free to reuse from here on
        h = torch.empty_like(self.u)
        M.moe_combine(s, self.u, self.y_perm, self.y_shared, self.w, self.slot_row, h)
        return h


def forward(rank_state: ExpertParallelRank, u: torch.Tensor, group=None) -> torch.Tensor:
    """One expert-parallel layer step on this rank (torch.distributed, one
    process per rank)."""
    r = rank_state
    send_counts = r.begin(u)
    recv_counts = exchange_counts(send_counts, r.world, r.device, group)
    send, ss, recv, rs = r.receive_counts(recv_counts)
    exchange_rows(recv, send, rs, ss, group)
    y_send, ys, y_recv, yr = r.experts()
    exchange_rows(y_recv, y_send, yr, ys, group)
    return r.finish()


def _virtual_all_to_all(recv: List[torch.Tensor], send: List[torch.Tensor],
                        recv_splits: List[List[int]], send_splits: List[List[int]]):
    """The row all-to-all between D ranks that live in one process: rank d's
    block for rank r lands in rank r's buffer at the offset of source d."""
    D = len(send)
    for d in range(D):
        src_off = np.concatenate([[0], np.cumsum(send_splits[d])])
        for r in range(D):
            dst_off = int(np.sum(recv_splits[r][:d]))
            n = int(send_splits[d][r])
            assert n == recv_splits[r][d]
            if n:
                recv[r][dst_off:dst_off + n].copy_(send[d][int(src_off[r]):int(src_off[r]) + n])


def forward_virtual(ranks: List[ExpertParallelRank], us: List[torch.Tensor]) -> List[torch.Tensor]:
    """One layer step of D expert-parallel ranks held in one process on one
    device; the exchanges are device-to-device copies."""
    D = len(ranks)
    el = ranks[0].el
    send_counts = [r.begin(u) for r, u in zip(ranks, us)]
    recv_counts = [np.concatenate([send_counts[s][d * el:(d + 1) * el] for s in range(D)])
                   for d in range(D)]
    bufs = [r.receive_counts(c) for r, c in zip(ranks, recv_counts)]
    _virtual_all_to_all([b[2] for b in bufs], [b[0] for b in bufs], [b[3] for b in bufs],
                        [b[1] for b in bufs])
    back = [r.experts() for r in ranks]
    _virtual_all_to_all([b[2] for b in back], [b[0] for b in back], [b[3] for b in back],
                        [b[1] for b in back])
    return [r.finish() for r in ranks]
