"""GPU grouping (moe_permute) against the oracle's stable counting sort:
offsets, perm_src, slot_row and x_perm bit-exact."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as orc
from tests.gpu_util import dev_bf16, dev_i32, host_bits, lib

pytestmark = pytest.mark.gpu


def run_permute(cfg, x_bits, ids):
    moe = lib()
    T, K, n = cfg.T, cfg.top_k, cfg.n_experts
    R = T * K
    offsets = torch.full((n + 1,), -5, dtype=torch.int32, device="cuda")
    perm_src = torch.full((max(R, 1),), -5, dtype=torch.int32, device="cuda")
    slot_row = torch.full((max(R, 1),), -5, dtype=torch.int32, device="cuda")
    x_perm = torch.zeros((max(R, 1), cfg.dim), dtype=torch.bfloat16, device="cuda")
    ws = moe.new_workspace(cfg)
    x = dev_bf16(x_bits) if T > 0 else torch.zeros((1, cfg.dim), dtype=torch.bfloat16, device="cuda")
    d_ids = dev_i32(ids) if T > 0 else torch.zeros((1, K), dtype=torch.int32, device="cuda")
    moe.moe_permute(cfg, x, d_ids, offsets, perm_src, slot_row, x_perm, ws)
    torch.cuda.synchronize()
    return (offsets.cpu().numpy(), perm_src[:R].cpu().numpy(), slot_row[:R].cpu().numpy(),
            host_bits(x_perm[:R]))


def check_permute(cfg, x_bits, ids):
    offsets, perm_src, slot_row, x_perm = run_permute(cfg, x_bits, ids)
    counts, r_off, r_src, r_slot = orc.routing_tables(ids, cfg.n_experts)
    assert np.array_equal(offsets, r_off)
    assert np.array_equal(perm_src, r_src)
    assert np.array_equal(slot_row, r_slot)
    assert np.array_equal(x_perm, x_bits[r_src])


def random_ids(rng, T, n, K, weights=None):
    if weights is None:
        return np.stack([rng.permutation(n)[:K] for _ in range(T)]).astype(np.int32)
    out = np.empty((T, K), np.int32)
    for t in range(T):
        out[t] = rng.choice(n, size=K, replace=False, p=weights)
    return out


# the grouping runs as one block up to 2048 assignments, one cluster up to
# 8192 (2049, 4096 + 2, 8192 below), and histogram / scan / scatter above
@pytest.mark.parametrize("T,n,K", [(1, 8, 2), (64, 8, 2), (129, 8, 2), (1000, 8, 2),
                                   (3000, 8, 2), (257, 1, 1), (300, 8, 8), (555, 32, 3),
                                   (100, 64, 6), (300, 256, 8), (2000, 160, 8), (5, 160, 8),
                                   (2049, 8, 1), (2049, 8, 2), (4096, 8, 2), (4097, 8, 2),
                                   (1024, 256, 8), (2730, 7, 3)])
def test_permute_matches_counting_sort(T, n, K):
    rng = np.random.default_rng(T * 31 + n)
    cfg = mi.Config("p", T=T, dim=128, hidden=128, n_experts=n, top_k=K, seed=900 + T)
    x = mi.gen_x(cfg)
    check_permute(cfg, x, random_ids(rng, T, n, K))


def test_permute_skewed_and_empty_experts():
    rng = np.random.default_rng(5)
    cfg = mi.Config("p", T=2049, dim=256, hidden=128, seed=77)
    w = np.array([0.7, 0.2, 0.1, 0, 0, 0, 0, 0])
    ids = random_ids(rng, cfg.T, 8, 2, np.where(w > 0, w, 0) / w.sum())
    check_permute(cfg, mi.gen_x(cfg), ids)


def test_permute_all_tokens_one_expert():
    cfg = mi.Config("p", T=700, dim=128, hidden=128, n_experts=4, top_k=1, seed=78)
    ids = np.full((700, 1), 2, np.int32)
    check_permute(cfg, mi.gen_x(cfg), ids)


def test_permute_all_assignments_one_expert_one_cluster():
    # 8192 assignments (the most the one-cluster grouping takes), all to expert 3
    cfg = mi.Config("p", T=8192, dim=128, hidden=128, n_experts=4, top_k=1, seed=79)
    ids = np.full((8192, 1), 3, np.int32)
    check_permute(cfg, mi.gen_x(cfg), ids)


def test_permute_zero_tokens():
    cfg = mi.Config("p", T=0, dim=128, hidden=128)
    offsets, *_ = run_permute(cfg, np.zeros((0, 128), np.uint16), np.zeros((0, 2), np.int32))
    assert np.all(offsets == 0)


def test_permute_full_size_skew():
    cfg = mi.CONFIGS["skew"]
    wg = mi.gen_router_weight(cfg)
    x = mi.gen_x(cfg, 0, mi.skew_shift(cfg, wg))
    ids, _, _ = orc.router(x, wg, cfg.top_k)
    check_permute(cfg, x, ids.astype(np.int32))
