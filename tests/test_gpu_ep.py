"""Expert parallelism on one GPU: two (or four) ranks' buffers in one
process, every arithmetic step in the CUDA library (router, grouping, the
grouped FFN of each rank's own experts, combine), the NCCL transfers replaced
by device copies that follow the same exchange plans.  Each rank's output is
compared with the fp64 oracle's whole layer on that rank's tokens.  (The
transfers themselves are exercised across processes by the gloo tests.)"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as orc
from tests.gpu_util import assert_bf16_close, dev_bf16, host_bits
from tests.inputs_filtered import filter_x

pytestmark = pytest.mark.gpu


def loopback(plans, send_bufs, recv_bufs, direction):
    """Device copies standing in for the point-to-point exchange of all ranks:
    direction 'dispatch' moves send chunks to the owners' receive chunks,
    'return' the reverse."""
    for src, p in enumerate(plans):
        for c in (p.send if direction == "dispatch" else p.recv):
            if c.count == 0:
                continue
            dst_plan = plans[c.peer]
            peer_chunks = dst_plan.recv if direction == "dispatch" else dst_plan.send
            d = [x for x in peer_chunks if x.peer == src and x.expert == c.expert]
            assert len(d) == 1 and d[0].count == c.count
            recv_bufs[c.peer][d[0].start:d[0].start + c.count].copy_(
                send_bufs[src][c.start:c.start + c.count])


def run_ep(world, tokens, dim, hidden, n, K, seed):
    from sparse_mixture_experts_46_b300.ep import ExpertParallelLayer
    nl = n // world
    cfg = mi.Config("ep", T=max(tokens), dim=dim, hidden=hidden, n_experts=n, top_k=K, seed=seed)
    L = mi.make_layer(cfg)
    xs = []
    for r in range(world):
        c = cfg.replace(T=max(tokens[r], 1), seed=seed + 1 + r)
        x = mi.gen_x(c)
        filter_x(c, x, L.wg)
        xs.append(x[:tokens[r]])
    wg = dev_bf16(L.wg)
    ranks = [ExpertParallelLayer(wg, dev_bf16(L.w1[r * nl:(r + 1) * nl]),
                                 dev_bf16(L.w3[r * nl:(r + 1) * nl]),
                                 dev_bf16(L.w2[r * nl:(r + 1) * nl]), K, r, world)
             for r in range(world)]
    xd = [dev_bf16(x) if len(x) else torch.empty((0, dim), dtype=torch.bfloat16, device="cuda")
          for x in xs]
    sts = [ranks[r].route(xd[r]) for r in range(world)]
    counts_all = torch.stack([st["counts"] for st in sts])
    plans = [ranks[r].plan(counts_all) for r in range(world)]
    bufs = [ranks[r].recv_buffers(plans[r], xd[r]) for r in range(world)]
    loopback(plans, [st["x_perm"] for st in sts], [b[0] for b in bufs], "dispatch")
    for r in range(world):
        ranks[r].ffn(plans[r], bufs[r][0], bufs[r][1])
    loopback(plans, [b[1] for b in bufs], [st["y_perm"] for st in sts], "return")
    ys = []
    for r in range(world):
        y = torch.full_like(xd[r], float("nan"))
        ranks[r].combine(sts[r], y)
        ys.append(y)
    torch.cuda.synchronize()
    for r in range(world):
        if tokens[r] == 0:
            continue
        ref, r_ids, _ = orc.moe_layer(xs[r], L.wg, L.w1, L.w3, L.w2, K)
        assert np.array_equal(np.sort(sts[r]["ids"].cpu().numpy(), 1), np.sort(r_ids, 1))
        assert_bf16_close(host_bits(ys[r]), ref, "rank %d layer output" % r)
    return plans


def test_two_ranks_mixtral_shaped():
    # 8 experts over 2 ranks at dim 4096: the owner's FFN runs on rows that
    # arrived from both ranks, grouped by its own experts
    plans = run_ep(2, [24, 40], 4096, 1024, 8, 2, 46800)
    assert all(p.recv_rows > 0 for p in plans)


def test_four_ranks_uneven_tokens_and_an_empty_rank():
    plans = run_ep(4, [300, 7, 0, 129], 256, 256, 8, 2, 46810)
    assert sum(p.recv_rows for p in plans) == 2 * (300 + 7 + 0 + 129)


def test_fine_grained_experts_over_two_ranks():
    run_ep(2, [200, 150], 256, 256, 160, 8, 46820)
