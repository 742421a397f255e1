"""Whole MoE layer on the GPU against the fp64 oracle, on the Mixtral-shaped
workloads: routing (ids, counts, offsets, permutation) bit-exact on every
token, outputs within |gpu - oracle| <= 1e-2 + 1e-2 |oracle| on every token
the oracle evaluates (all tokens of the small cases, a seeded sample at full
size), and the fused entry point bit-identical to the step-by-step calls."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as orc
from tests.gpu_util import assert_bf16_close, dev_bf16, host_bits, lib
from tests.inputs_filtered import filter_x

pytestmark = pytest.mark.gpu

_cache = {}


def layer(name):
    """Gap-filtered inputs of a named workload (or a Config), uploaded once per session."""
    if not isinstance(name, str):
        cfg = name
        name = cfg.name
        _cache.pop(name, None)
    else:
        cfg = mi.CONFIGS[name]
    if name not in _cache:
        _cache.clear()
        L = mi.make_layer(cfg)
        filter_x(cfg, L.x, L.wg, L.shift)
        dev = {k: dev_bf16(getattr(L, k)) for k in ("x", "wg", "w1", "w3", "w2")}
        _cache[name] = (cfg, L, dev)
    return _cache[name]


def stepwise(cfg, dev, path):
    """router -> permute -> expert FFN -> combine through the individual entry points."""
    moe = lib()
    T, K, n, d, h = cfg.T, cfg.top_k, cfg.n_experts, cfg.dim, cfg.hidden
    R = T * K
    i32 = dict(dtype=torch.int32, device="cuda")
    ids = torch.empty((T, K), **i32)
    gates = torch.empty((T, K), dtype=torch.float32, device="cuda")
    counts = torch.empty((n,), **i32)
    offsets = torch.empty((n + 1,), **i32)
    perm_src = torch.empty((R,), **i32)
    slot_row = torch.empty((R,), **i32)
    x_perm = torch.empty((R, d), dtype=torch.bfloat16, device="cuda")
    hbuf = torch.empty((R, h), dtype=torch.bfloat16, device="cuda")
    y_perm = torch.empty((R, d), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    ws = moe.new_workspace(cfg)
    moe.moe_router_topk(cfg, dev["x"], dev["wg"], ids, gates, counts)
    moe.moe_permute(cfg, dev["x"], ids, offsets, perm_src, slot_row, x_perm, ws)
    moe.moe_expert_ffn_grouped(cfg, x_perm, offsets, dev["w1"], dev["w3"], dev["w2"], hbuf,
                               y_perm, ws, path=path)
    moe.moe_combine(cfg, y_perm, slot_row, gates, y)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    out = dict(ids=ids, gates=gates, counts=counts, offsets=offsets, perm_src=perm_src,
               slot_row=slot_row, y=y)
    return {k: (host_bits(v) if v.dtype == torch.bfloat16 else v.cpu().numpy())
            for k, v in out.items()}


def fused(cfg, dev, path):
    moe = lib()
    y = torch.empty((cfg.T, cfg.dim), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    ws = moe.new_workspace(cfg)
    moe.moe_layer_forward(cfg, dev["x"], dev["wg"], dev["w1"], dev["w3"], dev["w2"], y, ws,
                          ids=ids, ffn_path=path)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    return host_bits(y), ids.cpu().numpy()


def check_layer(name, path, sample=None):
    cfg, L, dev = layer(name)
    name = cfg.name
    got = stepwise(cfg, dev, path)
    # routing: every token, bit-exact
    r_ids, r_gates, _ = orc.router(L.x, L.wg, cfg.top_k)
    assert np.array_equal(got["ids"], r_ids)
    assert np.max(np.abs(got["gates"] - r_gates)) < 1e-5
    counts, offsets, perm_src, slot_row = orc.routing_tables(r_ids, cfg.n_experts)
    assert np.array_equal(got["counts"], counts)
    assert np.array_equal(got["offsets"], offsets)
    assert np.array_equal(got["perm_src"], perm_src)
    assert np.array_equal(got["slot_row"], slot_row)
    # outputs: all tokens or a seeded sample, each token evaluated independently
    if sample is None:
        rows = np.arange(cfg.T)
    else:
        rows = np.sort(np.random.default_rng(cfg.seed).choice(cfg.T, sample, replace=False))
    ref, _, _ = orc.moe_layer(L.x[rows], L.wg, L.w1, L.w3, L.w2, cfg.top_k)
    assert_bf16_close(got["y"][rows], ref, "%s layer output" % name)
    # the fused entry point runs the same kernels: identical bits
    y_fused, ids_fused = fused(cfg, dev, path)
    assert np.array_equal(ids_fused, got["ids"])
    assert np.array_equal(y_fused, got["y"])


@pytest.mark.parametrize("path", [0, 1, 2])
def test_tiny_layer(path):
    check_layer("tiny", path)


@pytest.mark.parametrize("path", [0, 1])
def test_decode_layer_mixtral_dims(path):
    check_layer("decode", path)


def test_prefill_layer_mixtral_dims():
    check_layer("prefill", 0, sample=48)


def test_skewed_routing_layer():
    cfg, L, _ = layer("skew")
    ids, _, _ = orc.router(L.x, L.wg, cfg.top_k)
    share = np.bincount(ids[:, 0], minlength=8) / cfg.T
    assert 0.36 < share[0] < 0.50            # Zipf(1.2) top-1 share of the largest expert
    check_layer("skew", 0, sample=48)


@pytest.mark.parametrize("path", [0, 1, 2])
def test_fine_grained_layer_160_experts_top8(path):
    # "routing to, for example, 8 out of 160 much smaller experts"
    cfg = mi.Config("fine-small", T=600, dim=256, hidden=256, n_experts=160, top_k=8, seed=46107)
    check_layer(cfg, path)


def test_fine_grained_layer_full_dims_sampled():
    cfg = mi.CONFIGS["fine"].replace(T=1024)
    check_layer(cfg, 0, sample=32)


@pytest.mark.parametrize("path", [0, 3])
def test_mixtral_8x22b_dims(path):
    # "Mixtral 8x22B, scaling the exact same architecture up": dim 6144, hidden 16384
    cfg = mi.Config("8x22b", T=48, dim=6144, hidden=16384, seed=46108)
    check_layer(cfg, path)


def test_largest_batch_mixtral_dims_sampled():
    # T = 65536 at Mixtral dims: T * K * hidden = 1.88e9, just under the 2^31
    # limit of the supported shapes, so byte offsets into x_perm and H run far
    # past 2^31 and every expert's rows are walked in L2-sized blocks
    cfg = mi.CONFIGS["prefill"].replace(name="max-batch", T=65536, seed=46111)
    check_layer(cfg, 0, sample=32)
