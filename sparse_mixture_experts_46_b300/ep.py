"""Expert parallelism: the sparse MoE layer with its experts partitioned over
ranks ("Mixtral of Experts" section 2.1, the Expert Parallelism paragraph:
each device holds a subset of the experts, tokens are sent to the device of
the expert that processes them and the results are returned to their original
positions; the load on a device follows the routing, so it can be uneven).

Rank r of W owns the experts [r*n/W, (r+1)*n/W) and keeps its own tokens (data
parallel over tokens).  One layer call on rank r:

  1. route its tokens and group them by expert (moe_router_topk, moe_permute):
     the grouped rows of expert e are x_perm[offsets[e] : offsets[e+1]];
  2. share the per-expert row counts of every rank (all-gather of n ints);
  3. dispatch: the chunk of expert e goes to the rank owning e; the owner
     receives, for each of its experts in turn, the chunks of ranks 0..W-1,
     so the rows it receives are already grouped by its local experts;
  4. run the grouped SwiGLU FFN of its local experts on those rows
     (moe_expert_ffn_grouped);
  5. return: every output chunk goes back to the rank it came from, landing
     at the same grouped rows its inputs left from (y_perm);
  6. combine its tokens' expert outputs with their gates (moe_combine).

Every arithmetic step runs in the CUDA library; this module holds the host
side only: the exchange plan (a few prefix sums over the counts) and the
point-to-point transfers, posted as one batch per direction through
torch.distributed (NCCL on GPUs; peer rows move only through the collective
library).  The exchange is a parameter so that the multi-rank logic can be
exercised without several GPUs (gloo ranks on the CPU, or several ranks'
buffers in one process joined by device copies).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Chunk:
    """Rows [start, start + count) of a local buffer, exchanged with `peer`
    for expert `expert` (a global expert id)."""
    peer: int
    expert: int
    start: int
    count: int


class EPPlan:
    """Exchange plan of one rank, from every rank's per-expert row counts.

    counts_all[s][e]: rows of rank s's grouped batch routed to expert e
    (all ranks see the same [W, n] table).  Experts are owned in contiguous
    blocks of n / W.

    send:    chunks of this rank's grouped rows (x_perm / y_perm), one per
             expert e, to owner(e); start = offsets[e] of this rank.
    recv:    chunks of the owner-side buffer, expert-major: for each local
             expert, the rows of rank 0, then rank 1, ...
    local_offsets: [n_local + 1] row offsets of the local experts in the
             receive buffer (the grouping the FFN reads).
    """

    def __init__(self, counts_all, world: int, rank: int):
        c = np.asarray(counts_all, dtype=np.int64)
        if c.ndim != 2 or c.shape[0] != world:
            raise ValueError("counts_all must be [world, n_experts]")
        n = c.shape[1]
        if n % world != 0:
            raise ValueError("n_experts (%d) must be a multiple of the world size (%d)"
                             % (n, world))
        if np.any(c < 0):
            raise ValueError("negative row count")
        self.world, self.rank, self.n = world, rank, n
        self.n_local = n // world
        self.first_expert = rank * self.n_local
        mine = c[rank]
        offsets = np.concatenate([[0], np.cumsum(mine)])
        self.send = [Chunk(e // self.n_local, e, int(offsets[e]), int(mine[e])) for e in range(n)]
        self.send_rows = int(offsets[-1])
        recv, start = [], 0
        local_offsets = [0]
        for el in range(self.n_local):
            e = self.first_expert + el
            for s in range(world):
                recv.append(Chunk(s, e, start, int(c[s, e])))
                start += int(c[s, e])
            local_offsets.append(start)
        self.recv = recv
        self.recv_rows = start
        self.local_offsets = np.asarray(local_offsets, dtype=np.int32)

    def owner(self, expert: int) -> int:
        return expert // self.n_local


def exchange_p2p(send_chunks, recv_chunks, send_buf, recv_buf, rank, group=None):
    """Post every non-empty chunk as one batch of point-to-point transfers
    (torch.distributed.batch_isend_irecv) and wait for them.  Chunks with this
    rank as peer are copied locally.  Transfers between one pair of ranks are
    matched in posting order: both sides list them by expert id."""
    import torch.distributed as dist
    ops = []
    local_sends = [c for c in send_chunks if c.peer == rank and c.count > 0]
    local_recvs = [c for c in recv_chunks if c.peer == rank and c.count > 0]
    for c in send_chunks:
        if c.count > 0 and c.peer != rank:
            ops.append(dist.P2POp(dist.isend, send_buf[c.start:c.start + c.count], c.peer, group))
    for c in recv_chunks:
        if c.count > 0 and c.peer != rank:
            ops.append(dist.P2POp(dist.irecv, recv_buf[c.start:c.start + c.count], c.peer, group))
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()
    # this rank's own experts: the chunk moves within the rank
    by_expert = {c.expert: c for c in local_recvs}
    for c in local_sends:
        d = by_expert[c.expert]
        recv_buf[d.start:d.start + d.count].copy_(send_buf[c.start:c.start + c.count])


def all_gather_counts(counts, world, group=None):
    """[n] per-expert counts of this rank -> [world, n] of every rank."""
    import torch
    import torch.distributed as dist
    flat = torch.empty((world * counts.numel(),), dtype=counts.dtype, device=counts.device)
    dist.all_gather_into_tensor(flat, counts.reshape(-1).contiguous(), group=group)
    return flat.view(world, counts.numel())


class ExpertParallelLayer:
    """One rank's share of an expert-parallel MoE layer on the GPU.

    w_gate [dim, n] (replicated), w1/w3 [n_local, hidden, dim] and
    w2 [n_local, dim, hidden]: the weights of this rank's experts
    [rank * n_local, (rank + 1) * n_local).  forward(x) runs the six steps of
    the module docstring; its phases are also callable one by one (route,
    plan, recv_buffers, ffn, combine, with an exchange between them), which is
    how several ranks' buffers can be driven from one process with an
    exchange made of device copies."""

    def __init__(self, w_gate, w1, w3, w2, top_k, rank, world, group=None):
        self.w_gate, self.w1, self.w3, self.w2 = w_gate, w1, w3, w2
        self.dim, self.n = w_gate.shape
        self.hidden = w1.shape[1]
        self.n_local = w1.shape[0]
        if self.n_local * world != self.n:
            raise ValueError("each rank holds n / world experts")
        self.top_k, self.rank, self.world, self.group = top_k, rank, world, group

    # -- phase 1: routing and grouping of this rank's tokens (library kernels)
    def route(self, x):
        import torch
        import sparse_mixture_experts_46_b300 as moe
        T, K, n, d = x.shape[0], self.top_k, self.n, self.dim
        R = T * K
        dev = x.device
        s = moe.make_shape(T, d, self.hidden, n, K)
        i32 = dict(dtype=torch.int32, device=dev)
        st = dict(shape=s, T=T, ids=torch.empty((T, K), **i32),
                  gates=torch.empty((T, K), dtype=torch.float32, device=dev),
                  counts=torch.empty((n,), **i32), offsets=torch.empty((n + 1,), **i32),
                  perm_src=torch.empty((R,), **i32), slot_row=torch.empty((R,), **i32),
                  x_perm=torch.empty((R, d), dtype=x.dtype, device=dev),
                  y_perm=torch.empty((R, d), dtype=x.dtype, device=dev))
        ws = moe.new_workspace(s, device=dev)
        moe.moe_router_topk(s, x, self.w_gate, st["ids"], st["gates"], st["counts"])
        moe.moe_permute(s, x, st["ids"], st["offsets"], st["perm_src"], st["slot_row"],
                        st["x_perm"], ws)
        return st

    # -- phase 2: the exchange plan from every rank's counts
    def plan(self, counts_all):
        return EPPlan(counts_all.cpu().numpy() if hasattr(counts_all, "cpu") else counts_all,
                      self.world, self.rank)

    # -- phase 3 buffers: rows this rank receives for its experts
    def recv_buffers(self, plan, like):
        import torch
        return (torch.empty((plan.recv_rows, self.dim), dtype=like.dtype, device=like.device),
                torch.empty((plan.recv_rows, self.dim), dtype=like.dtype, device=like.device))

    # -- phase 4: the grouped FFN of the local experts on the received rows
    def ffn(self, plan, x_recv, y_recv):
        import torch
        import sparse_mixture_experts_46_b300 as moe
        R = plan.recv_rows
        if R == 0:
            return
        s = moe.make_shape(R, self.dim, self.hidden, self.n_local, 1)
        offs = torch.as_tensor(plan.local_offsets, dtype=torch.int32).to(x_recv.device)
        h = torch.empty((R, self.hidden), dtype=x_recv.dtype, device=x_recv.device)
        ws = moe.new_workspace(s, device=x_recv.device)
        moe.moe_expert_ffn_grouped(s, x_recv, offs, self.w1, self.w3, self.w2, h, y_recv, ws)
        status = moe.moe_check_error(ws)
        if status != moe.MOE_OK:
            raise moe.MoeError(status, "moe_expert_ffn_grouped (expert-parallel)")

    # -- phase 6: gated combine (library kernel)
    def combine(self, st, y):
        import sparse_mixture_experts_46_b300 as moe
        moe.moe_combine(st["shape"], st["y_perm"], st["slot_row"], st["gates"], y)

    def forward(self, x, y=None, exchange=exchange_p2p):
        """The whole layer on this rank, with torch.distributed collectives."""
        import torch
        st = self.route(x)
        counts_all = all_gather_counts(st["counts"], self.world, self.group)
        plan = self.plan(counts_all)
        x_recv, y_recv = self.recv_buffers(plan, x)
        exchange(plan.send, plan.recv, st["x_perm"], x_recv, self.rank, self.group)
        self.ffn(plan, x_recv, y_recv)
        exchange(plan.recv, plan.send, y_recv, st["y_perm"], self.rank, self.group)
        if y is None:
            y = torch.empty_like(x)
        self.combine(st, y)
        return y
