"""GPU router (moe_router_topk) against the fp64 oracle: ids and counts
bit-exact, gates within 1e-5, on inputs whose selection is gap-filtered (a
token whose two selected logits are within 1e-4 of each other keeps its
place and has its ids compared as a set)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as orc
from tests.gpu_util import dev_bf16, lib
from tests.inputs_filtered import check_routing, filter_x, order_decided

pytestmark = pytest.mark.gpu


def run_router(cfg, x_bits, wg_bits):
    moe = lib()
    T, K, n = cfg.T, cfg.top_k, cfg.n_experts
    ids = torch.full((max(T, 1), K), -7, dtype=torch.int32, device="cuda")
    gates = torch.full((max(T, 1), K), -7.0, dtype=torch.float32, device="cuda")
    counts = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    x = dev_bf16(x_bits) if T > 0 else torch.empty((1, cfg.dim), dtype=torch.bfloat16, device="cuda")
    moe.moe_router_topk(cfg, x, dev_bf16(wg_bits), ids, gates, counts)
    torch.cuda.synchronize()
    return ids[:T].cpu().numpy(), gates[:T].cpu().numpy(), counts.cpu().numpy()


def check_router(cfg, x_bits, wg_bits):
    ids, gates, counts = run_router(cfg, x_bits, wg_bits)
    r_ids, r_gates, _ = orc.router(x_bits, wg_bits, cfg.top_k)
    check_routing(ids, gates, r_ids, r_gates, order_decided(x_bits, wg_bits, cfg.top_k))
    assert np.array_equal(counts, np.bincount(r_ids.reshape(-1), minlength=cfg.n_experts))


def layer_inputs(cfg):
    x = mi.gen_x(cfg)
    wg = mi.gen_router_weight(cfg)
    filter_x(cfg, x, wg)
    return x, wg


@pytest.mark.parametrize("T,dim,n,K", [
    (64, 128, 8, 2), (1, 128, 8, 2), (2, 256, 8, 2), (127, 128, 8, 2), (129, 384, 8, 2),
    (300, 128, 1, 1), (200, 128, 8, 8), (200, 128, 5, 3), (150, 256, 16, 2), (100, 128, 32, 4),
    (77, 128, 12, 1),
    # batches of >= 512 tokens take the warp router (W_g staged in shared memory)
    (513, 256, 8, 2), (1000, 384, 5, 3), (600, 128, 16, 2), (777, 256, 12, 1),
    (512, 128, 8, 8), (1030, 512, 16, 16), (2049, 4096, 8, 2),
    # more than 32 experts (fine-grained MoE): the wide tensor-core router
    (200, 256, 40, 2), (1000, 512, 64, 6), (700, 256, 160, 8), (129, 128, 256, 8),
    (1, 256, 160, 8), (64, 128, 48, 1), (600, 4096, 160, 8),
    # the wide router splits the model dimension over a cluster of up to 8 CTAs
    # while the token tiles leave SMs idle; 75 tiles (9600 tokens) run unsplit
    (16, 4096, 160, 8), (9600, 128, 40, 2),
    # Mixtral's model dimension and half of it: single tokens, fewer tokens
    # than SMs, fewer than 8 experts, K = n, and 20000 tokens
    (1, 4096, 8, 2), (16, 4096, 8, 2), (77, 2048, 8, 2), (300, 4096, 5, 3),
    (129, 4096, 1, 1), (1000, 2048, 8, 8), (20000, 4096, 8, 2), (4097, 2048, 7, 1)])
def test_router_matches_oracle(T, dim, n, K):
    cfg = mi.Config("r", T=T, dim=dim, hidden=128, n_experts=n, top_k=K, seed=700 + T + n)
    x, wg = layer_inputs(cfg)
    check_router(cfg, x, wg)


def test_router_exact_ties_go_to_lower_index():
    cfg = mi.Config("tie", T=33, dim=128, hidden=128)
    x = np.zeros((33, 128), np.uint16)      # all logits exactly 0
    wg = mi.gen_router_weight(cfg)
    ids, gates, counts = run_router(cfg, x, wg)
    assert np.all(ids == np.array([0, 1]))
    assert np.all(gates == 0.5)
    assert counts.tolist() == [33, 33, 0, 0, 0, 0, 0, 0]


@pytest.mark.parametrize("dim", [128, 4096])
def test_router_exact_ties_go_to_lower_index_at_dims(dim):
    # all logits exactly 0, at a small and at Mixtral's model dimension
    cfg = mi.Config("tie", T=300, dim=dim, hidden=128)
    x = np.zeros((cfg.T, dim), np.uint16)
    ids, gates, counts = run_router(cfg, x, mi.gen_router_weight(cfg))
    assert np.all(ids == np.array([0, 1]))
    assert np.all(gates == 0.5)
    assert counts.tolist() == [cfg.T, cfg.T, 0, 0, 0, 0, 0, 0]


def test_warp_router_exact_ties_go_to_lower_index():
    cfg = mi.Config("tie", T=1025, dim=256, hidden=128, n_experts=16, top_k=3)
    x = np.zeros((cfg.T, cfg.dim), np.uint16)
    ids, gates, counts = run_router(cfg, x, mi.gen_router_weight(cfg))
    assert np.all(ids == np.array([0, 1, 2]))
    assert np.allclose(gates, 1.0 / 3.0, rtol=0, atol=1e-7)
    assert counts.tolist() == [cfg.T] * 3 + [0] * 13


def test_wide_router_exact_ties_go_to_lower_index():
    cfg = mi.Config("tie", T=300, dim=256, hidden=128, n_experts=160, top_k=8)
    x = np.zeros((cfg.T, cfg.dim), np.uint16)
    ids, gates, counts = run_router(cfg, x, mi.gen_router_weight(cfg))
    assert np.all(ids == np.arange(8))
    assert np.allclose(gates, 1.0 / 8.0, rtol=0, atol=1e-7)
    assert counts.tolist() == [cfg.T] * 8 + [0] * 152


@pytest.mark.parametrize("n,K,dim", [(8, 2, 128), (24, 2, 128), (40, 4, 128), (8, 2, 4096)])
def test_router_nan_logit_counts_as_minus_infinity(n, K, dim):
    # every token's logit for expert 3 is NaN (a NaN column of W_g): all three
    # routers (tensor-core n <= 16, CUDA-core n <= 32, wide) must route as if
    # expert 3 did not exist, at a small and at Mixtral's model dimension
    cfg = mi.Config("nan", T=200, dim=dim, hidden=128, n_experts=n, top_k=K, seed=900 + n)
    wg = mi.gen_router_weight(cfg)
    keep = [e for e in range(n) if e != 3]
    wg_rest = np.ascontiguousarray(wg[:, keep])
    x = mi.gen_x(cfg)
    filter_x(cfg.replace(n_experts=n - 1), x, wg_rest)
    wg_nan = wg.copy()
    wg_nan[:, 3] = 0x7FC0                   # bf16 quiet NaN
    ids, gates, counts = run_router(cfg, x, wg_nan)
    r_ids, r_gates, _ = orc.router(x, wg_rest, K)
    check_routing(ids, gates, np.where(r_ids >= 3, r_ids + 1, r_ids), r_gates,
                  order_decided(x, wg_rest, K))
    assert counts[3] == 0


def test_router_zero_tokens_clears_counts():
    cfg = mi.Config("empty", T=0, dim=128, hidden=128)
    _, _, counts = run_router(cfg, np.zeros((0, 128), np.uint16), mi.gen_router_weight(cfg))
    assert np.all(counts == 0)


@pytest.mark.parametrize("name", ["prefill", "skew"])
def test_router_full_size(name):
    cfg = mi.CONFIGS[name]
    wg = mi.gen_router_weight(cfg)
    shift = mi.skew_shift(cfg, wg) if cfg.zipf_s > 0 else None
    x = mi.gen_x(cfg, 0, shift)
    filter_x(cfg, x, wg, shift)
    check_router(cfg, x, wg)
