"""Expert parallelism (sparse_mixture_experts_46_b300.ep) on the CPU: the
exchange plan's arithmetic, and the whole dispatch / expert FFN / return /
combine path run by gloo ranks, each rank's layer output compared with the
fp64 oracle's layer on that rank's tokens.  The arithmetic steps here are the
oracle's (routing, grouping, grouped FFN, combine); what is under test is the
plan and the point-to-point exchange that the GPU path uses unchanged."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plan_chunks_are_consistent_across_ranks():
    from sparse_mixture_experts_46_b300.ep import EPPlan
    # 3 ranks, 6 experts (2 per rank); rank 2 routed nothing to expert 5
    counts = np.array([[3, 0, 2, 5, 1, 4],
                       [0, 7, 1, 1, 2, 2],
                       [4, 4, 0, 3, 6, 0]])
    plans = [EPPlan(counts, 3, r) for r in range(3)]
    for r, p in enumerate(plans):
        assert p.n_local == 2 and p.first_expert == 2 * r
        # send chunks tile this rank's grouped rows, expert by expert
        assert [c.start for c in p.send] == list(np.concatenate([[0], np.cumsum(counts[r])[:-1]]))
        assert [c.peer for c in p.send] == [0, 0, 1, 1, 2, 2]
        assert p.send_rows == counts[r].sum()
        # receive chunks: expert-major, ranks ascending inside each expert
        assert [(c.expert, c.peer) for c in p.recv] == [(2 * r + el, s) for el in range(2)
                                                         for s in range(3)]
        assert p.recv_rows == counts[:, 2 * r:2 * r + 2].sum()
        assert list(p.local_offsets) == [0, counts[:, 2 * r].sum(), p.recv_rows]
    # every send chunk (src -> dst, expert e) meets a receive chunk of the same size
    for src, p in enumerate(plans):
        for c in p.send:
            match = [d for d in plans[c.peer].recv if d.peer == src and d.expert == c.expert]
            assert len(match) == 1 and match[0].count == c.count


def test_plan_rejects_uneven_expert_split():
    from sparse_mixture_experts_46_b300.ep import EPPlan
    with pytest.raises(ValueError):
        EPPlan(np.zeros((3, 8), dtype=int), 3, 0)
    with pytest.raises(ValueError):
        EPPlan(np.full((2, 8), -1), 2, 0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _layer_inputs(world, rank, tokens, skew):
    import moe_inputs as mi
    # same weights on every rank (same seed), rank-specific tokens
    cfg = mi.Config("ep", T=max(tokens[rank], 1), dim=32, hidden=48, n_experts=4 * world,
                    top_k=2, seed=46700)
    L = mi.make_layer(cfg)
    x = mi.gen_x(cfg.replace(seed=46710 + rank))[:tokens[rank]]
    if skew:
        # push every token toward the last rank's experts: a shift along the
        # router columns of those experts (load imbalance across ranks)
        from oracle import moe_oracle as orc
        wg = orc.widen_bf16(L.wg)
        push = wg[:, -4:].sum(axis=1)
        xf = orc.widen_bf16(x) + 2.0 * push / np.linalg.norm(push)
        x = orc.round_bf16(xf)
    return cfg, L, x


def _rank(rank, world, port, tokens, skew, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import moe_oracle as orc
    from sparse_mixture_experts_46_b300.ep import EPPlan, all_gather_counts, exchange_p2p
    cfg, L, x = _layer_inputs(world, rank, tokens, skew)
    K, n = cfg.top_k, cfg.n_experts
    nl = n // world
    # 1. route and group (oracle arithmetic)
    ids, gates, _ = orc.router(x, L.wg, K)
    counts, offsets, perm_src, slot_row = orc.routing_tables(ids, n)
    x_perm = torch.from_numpy(orc.widen_bf16(x)[perm_src].reshape(-1, cfg.dim))
    # 2. every rank's counts
    counts_all = all_gather_counts(torch.from_numpy(counts.astype(np.int64)), world)
    plan = EPPlan(counts_all.numpy(), world, rank)
    # 3. dispatch
    x_recv = torch.empty((plan.recv_rows, cfg.dim), dtype=torch.float64)
    exchange_p2p(plan.send, plan.recv, x_perm, x_recv, rank)
    # 4. the local experts' FFN on the received rows
    sl = slice(rank * nl, (rank + 1) * nl)
    y_recv, _ = orc.grouped_ffn(x_recv.numpy(), plan.local_offsets, L.w1[sl], L.w3[sl], L.w2[sl])
    # 5. return
    y_perm = torch.empty((plan.send_rows, cfg.dim), dtype=torch.float64)
    exchange_p2p(plan.recv, plan.send, torch.from_numpy(np.ascontiguousarray(y_recv)), y_perm,
                 rank)
    # 6. combine, against the whole layer on this rank's tokens
    y = orc.combine(y_perm.numpy(), slot_row, gates)
    ref, _, _ = orc.moe_layer(x, L.wg, L.w1, L.w3, L.w2, K)
    err = float(np.max(np.abs(y - ref), initial=0.0))
    out[rank] = (err, float(np.max(np.abs(ref), initial=0.0)), plan.recv_rows,
                 int(counts.sum()))
    dist.destroy_process_group()


def _run(world, tokens, skew=False):
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), tokens, skew, out), nprocs=world, join=True)
        return dict(out)


def test_two_ranks_match_the_whole_layer():
    res = _run(2, [40, 57])
    for rank, (err, scale, recv_rows, sent) in res.items():
        assert err <= 1e-12 * max(scale, 1.0), (rank, err)
    # every assignment was processed exactly once somewhere
    assert sum(r[2] for r in res.values()) == sum(r[3] for r in res.values()) == 2 * (40 + 57)


def test_four_ranks_skewed_load_and_an_empty_rank():
    # every token leans toward the last rank's experts, and rank 2 has no tokens
    res = _run(4, [30, 25, 0, 33], skew=True)
    for rank, (err, scale, recv_rows, sent) in res.items():
        assert err <= 1e-12 * max(scale, 1.0), (rank, err)
    assert res[2][3] == 0
    loads = [res[r][2] for r in range(4)]
    assert loads[3] == max(loads) and loads[3] > sum(loads) / 4   # the imbalance is real
    assert sum(loads) == 2 * (30 + 25 + 0 + 33)
