"""GPU routing statistics (moe_routing_stats) against the oracle's plain
restatement of section 5 of "Mixtral of Experts" (Fig. 7 / Fig. 9 counts per
expert and choice, Table 5 repeat counts): integer counts, bit-exact."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as orc
from tests.gpu_util import dev_bf16, dev_i32, lib

pytestmark = pytest.mark.gpu


def run_stats(cfg, ids):
    moe = lib()
    K, n = cfg.top_k, cfg.n_experts
    slot_counts = torch.full((K * n,), -3, dtype=torch.int32, device="cuda")
    repeats = torch.full((2,), -3, dtype=torch.int32, device="cuda")
    d_ids = dev_i32(ids) if cfg.T > 0 else torch.zeros((1, K), dtype=torch.int32, device="cuda")
    moe.moe_routing_stats(cfg, d_ids, slot_counts, repeats)
    torch.cuda.synchronize()
    return slot_counts.cpu().numpy().reshape(K, n), repeats.cpu().numpy()


def check(cfg, ids):
    counts, rep = run_stats(cfg, ids)
    ref = orc.routing_stats(ids, cfg.n_experts)
    assert np.array_equal(counts, ref["slot_counts"])
    assert rep.tolist() == [ref["first_repeat"], ref["any_repeat"]]


@pytest.mark.parametrize("T,n,K", [(1, 8, 2), (2, 8, 2), (1000, 8, 2), (7777, 8, 1), (300, 8, 8),
                                   (2000, 160, 8), (513, 32, 4)])
def test_stats_random_ids(T, n, K):
    rng = np.random.default_rng(T + n + K)
    ids = np.stack([rng.permutation(n)[:K] for _ in range(T)]).astype(np.int32)
    # runs of repeated choices, as consecutive tokens of real text show
    for t in range(1, T, 3):
        ids[t] = ids[t - 1]
    check(mi.Config("s", T=T, dim=128, hidden=128, n_experts=n, top_k=K), ids)


def test_stats_zero_tokens():
    cfg = mi.Config("s", T=0, dim=128, hidden=128)
    counts, rep = run_stats(cfg, np.zeros((0, 2), np.int32))
    assert not counts.any() and rep.tolist() == [0, 0]


def test_stats_of_the_router_on_the_prefill_batch():
    """The statistic on the GPU router's own ids for the Mixtral prefill batch
    (iid synthetic tokens: shares near 1/8, repeats near the random rates)."""
    moe = lib()
    cfg = mi.CONFIGS["prefill"]
    L = mi.make_layer(cfg, experts=False)
    ids = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    gates = torch.empty((cfg.T, cfg.top_k), dtype=torch.float32, device="cuda")
    counts = torch.empty((cfg.n_experts,), dtype=torch.int32, device="cuda")
    moe.moe_router_topk(cfg, dev_bf16(L.x), dev_bf16(L.wg), ids, gates, counts)
    h_ids = ids.cpu().numpy()
    check(cfg, h_ids)
    sc, rep = run_stats(cfg, h_ids)
    assert np.array_equal(sc.sum(0), counts.cpu().numpy())
    assert abs(rep[0] / (cfg.T - 1) - 0.125) < 0.03
    assert abs(rep[1] / (cfg.T - 1) - (1 - (6 / 8) * (5 / 7))) < 0.05
