"""Residual MoE stack x <- x + MoE_l(RMSNorm(x)) on the GPU (moe_layer_forward
with RMSNorm and residual), checked layer by layer against the fp64 oracle
with teacher forcing: the oracle takes the GPU's bf16 input of each layer.

Routing after the first layer is not gap-filtered, so the selected experts
are compared bit-exactly on the tokens whose oracle logits (on RMSNorm(x))
decide the selection by the gap filter's margin, their slot order where that
is decided too; the other tokens are counted.  Layer outputs must be within
|gpu - oracle| <= 1e-2 + 1e-2 |oracle| on every token routed like the oracle.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as orc
from tests.gpu_util import assert_bf16_close, dev_bf16, host_bits, lib
from tests.inputs_filtered import align_slots, ambiguous_tokens, order_decided

pytestmark = pytest.mark.gpu


def filter_first_layer(cfg, x, wg):
    """Gap filter on RMSNorm(x) for the first layer's router."""
    for attempt in range(1, 65):
        bad = ambiguous_tokens(orc.rmsnorm_bf16(x, cfg.rmsnorm_eps), wg, cfg.top_k)
        if not bad.any():
            return
        rows = np.nonzero(bad)[0]
        x[rows] = mi.gen_x_rows(cfg, rows, attempt)
    raise RuntimeError("gap filter did not converge")


def run_stack(cfg, rows):
    """Upload every layer, run the stack, then check each layer on `rows`."""
    moe = lib()
    x0 = mi.gen_x(cfg)
    filter_first_layer(cfg, x0, mi.gen_router_weight(cfg, 0))
    layers = []
    for l in range(cfg.layers):
        wg = mi.gen_router_weight(cfg, l)
        w1, w3, w2 = mi.gen_experts(cfg, l)
        layers.append(tuple(dev_bf16(a) for a in (wg, w1, w3, w2)))
        del w1, w3, w2
    xs = [dev_bf16(x0)]
    ids = []
    ws = moe.new_workspace(cfg)
    for l, (wg, w1, w3, w2) in enumerate(layers):
        y = torch.empty_like(xs[-1])
        i = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
        moe.moe_layer_forward(cfg, xs[-1], wg, w1, w3, w2, y, ws, ids=i,
                              rmsnorm_eps=cfg.rmsnorm_eps, residual=xs[-1])
        xs.append(y)
        ids.append(i)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    host_x = [host_bits(x[rows]) for x in xs]
    host_ids = [i[rows].cpu().numpy() for i in ids]
    del layers, xs
    torch.cuda.empty_cache()

    excluded = 0
    for l in range(cfg.layers):
        wg = mi.gen_router_weight(cfg, l)
        w1, w3, w2 = mi.gen_experts(cfg, l)
        ref, r_ids, _, u = orc.stack_layer(host_x[l], wg, w1, w3, w2, cfg.top_k, cfg.rmsnorm_eps)
        ok = ~ambiguous_tokens(u, wg, cfg.top_k)
        excluded += int((~ok).sum())
        align_slots(host_ids[l][ok], r_ids[ok], order_decided(u, wg, cfg.top_k)[ok])
        same = np.all(np.sort(host_ids[l], axis=1) == np.sort(r_ids, axis=1), axis=1)
        assert_bf16_close(host_x[l + 1][same], ref[same], "layer %d output" % l)
    return excluded


def test_tiny_stack_all_tokens():
    cfg = mi.CONFIGS["stack"].replace(T=96, dim=128, hidden=256, layers=4, seed=46105)
    excluded = run_stack(cfg, np.arange(cfg.T))
    assert excluded < cfg.T * cfg.layers // 4


def test_stack_warp_router_all_tokens():
    # >= 512 tokens: the RMSNorm is fused into the warp router
    cfg = mi.CONFIGS["stack"].replace(T=640, dim=256, hidden=256, layers=3, seed=46106)
    excluded = run_stack(cfg, np.arange(cfg.T))
    assert excluded < cfg.T * cfg.layers // 4


@pytest.mark.slow
def test_full_stack_sampled_tokens():
    cfg = mi.CONFIGS["stack"]
    rows = np.sort(np.random.default_rng(cfg.seed).choice(cfg.T, 256, replace=False))
    excluded = run_stack(cfg, rows)
    print("stack: %d of %d checked token-layers excluded from the routing comparison"
          % (excluded, 256 * cfg.layers))
