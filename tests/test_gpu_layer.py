"""Whole MoE layer on the GPU against the fp64 oracle, on the Mixtral-shaped
workloads: routing (ids, counts, offsets, permutation) bit-exact on every
token, outputs within |gpu - oracle| <= 1e-2 + 1e-2 |oracle| on every token
the oracle evaluates, for the step-by-step calls and for the fused entry
point.  Where both route with the same kernels (every batch but the
decode-sized one, which moe_layer_forward routes, groups and gathers in one
launch) the two are also bit-identical.

Which tokens the oracle evaluates: all of them, in every case here, so every
output element of the layer is compared -- including the Mixtral prefill layer
(T=4096), the skewed batch (T=16384) and the largest supported batch
(T=65536).  ``check_layer(..., sample=k)`` instead takes a stratified sample
(``tile_sample``) that puts checked rows in EVERY
256-row token tile of EVERY expert group -- the first and last row of each
tile and the two rows on either side of the split between the two CTAs of the
pair that computes it, so each expert's last, partial tile is always covered
-- plus a few seeded random tokens.  Every checked row is compared in full,
i.e. under every weight tile of both GEMMs.

Every output buffer of the step-by-step path, and the workspace, is the head
of a larger buffer whose tail holds a sentinel that must survive the call
(a write past the end of a buffer changes it)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as orc
from tests.gpu_util import Guarded, assert_bf16_close, dev_bf16, guarded_workspace, host_bits, lib
from tests.inputs_filtered import (aligned_slot_rows, check_routing, filter_x, order_decided,
                                   tile_sample)

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
    """router -> permute -> expert FFN -> combine through the individual entry
    points, every output canary-guarded and NaN / sentinel filled."""
    moe = lib()
    T, K, n, d, h = cfg.T, cfg.top_k, cfg.n_experts, cfg.dim, cfg.hidden
    R = T * K
    bufs = dict(ids=Guarded((T, K), torch.int32, -7), gates=Guarded((T, K), torch.float32, -7.0),
                counts=Guarded((n,), torch.int32, -7), offsets=Guarded((n + 1,), torch.int32, -7),
                perm_src=Guarded((R,), torch.int32, -7), slot_row=Guarded((R,), torch.int32, -7),
                x_perm=Guarded((R, d), torch.bfloat16, float("nan")),
                h=Guarded((R, h), torch.bfloat16, float("nan")),
                y_perm=Guarded((R, d), torch.bfloat16, float("nan")),
                y=Guarded((T, d), torch.bfloat16, float("nan")))
    v = {k: b.view for k, b in bufs.items()}
    ws, wsg = guarded_workspace(moe, cfg)
    moe.moe_router_topk(cfg, dev["x"], dev["wg"], v["ids"], v["gates"], v["counts"])
    moe.moe_permute(cfg, dev["x"], v["ids"], v["offsets"], v["perm_src"], v["slot_row"],
                    v["x_perm"], ws)
    moe.moe_expert_ffn_grouped(cfg, v["x_perm"], v["offsets"], dev["w1"], dev["w3"], dev["w2"],
                               v["h"], v["y_perm"], ws, path=path)
    moe.moe_combine(cfg, v["y_perm"], v["slot_row"], v["gates"], v["y"])
    assert moe.moe_check_error(ws) == moe.MOE_OK
    for k, b in bufs.items():
        b.check(k)
    wsg.check("workspace")
    out = {k: v[k] for k in ("ids", "gates", "counts", "offsets", "perm_src", "slot_row", "y")}
    return {k: (host_bits(t) if t.dtype == torch.bfloat16 else t.cpu().numpy())
            for k, t in out.items()}


def fused(cfg, dev, path):
    moe = lib()
    y = Guarded((cfg.T, cfg.dim), torch.bfloat16, float("nan"))
    ids = Guarded((cfg.T, cfg.top_k), torch.int32, -7)
    gates = Guarded((cfg.T, cfg.top_k), torch.float32, -7.0)
    ws, wsg = guarded_workspace(moe, cfg)
    moe.moe_layer_forward(cfg, dev["x"], dev["wg"], dev["w1"], dev["w3"], dev["w2"], y.view, ws,
                          ids=ids.view, gates=gates.view, ffn_path=path)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    y.check("y (fused)")
    ids.check("ids (fused)")
    gates.check("gates (fused)")
    wsg.check("workspace (fused)")
    return host_bits(y.view), ids.view.cpu().numpy(), gates.view.cpu().numpy()


def fused_routes_in_one_launch(cfg):
    """moe_layer_forward's decode-sized routing kernel: T <= 32, n <= 8."""
    return cfg.T <= 32 and cfg.n_experts <= 8


def check_layer(name, path, sample=None):
    """sample=None: every token; else a stratified per-tile sample plus
    `sample` seeded random tokens."""
    cfg, L, dev = layer(name)
    name = cfg.name
    got = stepwise(cfg, dev, path)
    # routing: every token, bit-exact (slot order compared where it is decided)
    r_ids, r_gates, _ = orc.router(L.x, L.wg, cfg.top_k)
    decided = order_decided(L.x, L.wg, cfg.top_k)
    p = check_routing(got["ids"], got["gates"], r_ids, r_gates, decided)
    counts, offsets, perm_src, slot_row = orc.routing_tables(r_ids, cfg.n_experts)
    assert np.array_equal(got["counts"], counts)
    assert np.array_equal(got["offsets"], offsets)
    assert np.array_equal(got["perm_src"], perm_src)
    assert np.array_equal(aligned_slot_rows(got["slot_row"], p), slot_row)
    # outputs: all tokens, or every token tile of every expert plus random tokens
    if sample is None:
        rows = np.arange(cfg.T)
    else:
        rnd = np.random.default_rng(cfg.seed).choice(cfg.T, sample, replace=False)
        rows = np.union1d(tile_sample(offsets, perm_src), rnd)
    ref, _, _ = orc.moe_layer(L.x[rows], L.wg, L.w1, L.w3, L.w2, cfg.top_k)
    assert_bf16_close(got["y"][rows], ref, "%s layer output" % name)
    # the fused entry point
    y_fused, ids_fused, gates_fused = fused(cfg, dev, path)
    check_routing(ids_fused, gates_fused, r_ids, r_gates, decided)
    if fused_routes_in_one_launch(cfg):
        assert_bf16_close(y_fused[rows], ref, "%s fused layer output" % name)
    else:
        # the same kernels: identical bits
        assert np.array_equal(ids_fused, got["ids"])
        assert np.array_equal(y_fused, got["y"])
    return rows


@pytest.mark.parametrize("path", [0, 1, 2])
def test_tiny_layer(path):
    check_layer("tiny", path)


@pytest.mark.parametrize("path", [0, 1])
def test_decode_layer_mixtral_dims(path):
    check_layer("decode", path)


def test_prefill_layer_mixtral_dims():
    # every token of the layer (the fp64 oracle takes a few seconds per expert)
    rows = check_layer("prefill", 0)
    assert len(rows) == mi.CONFIGS["prefill"].T


def test_skewed_routing_layer():
    cfg, L, _ = layer("skew")
    ids, _, _ = orc.router(L.x, L.wg, cfg.top_k)
    share = np.bincount(ids[:, 0], minlength=8) / cfg.T
    assert 0.36 < share[0] < 0.50            # Zipf(1.2) top-1 share of the largest expert
    check_layer("skew", 0)                   # every token


@pytest.mark.parametrize("path", [0, 1, 2])
def test_fine_grained_layer_160_experts_top8(path):
    # "routing to, for example, 8 out of 160 much smaller experts"
    cfg = mi.Config("fine-small", T=600, dim=256, hidden=256, n_experts=160, top_k=8, seed=46107)
    check_layer(cfg, path)


def test_fine_grained_layer_full_dims():
    cfg = mi.CONFIGS["fine"].replace(T=1024)
    check_layer(cfg, 0)


@pytest.mark.parametrize("path", [0, 3])
def test_mixtral_8x22b_dims(path):
    # "Mixtral 8x22B, scaling the exact same architecture up": dim 6144, hidden 16384
    cfg = mi.Config("8x22b", T=48, dim=6144, hidden=16384, seed=46108)
    check_layer(cfg, path)


@pytest.mark.parametrize("T,dim,n,K", [
    (1, 128, 8, 2), (32, 128, 8, 2), (17, 256, 8, 8), (9, 384, 5, 3), (32, 512, 1, 1),
    (20, 128, 8, 1), (31, 4096, 8, 2), (12, 6144, 6, 2), (7, 6144, 8, 2), (32, 256, 8, 8)])
def test_decode_sized_layer_routed_in_one_launch(T, dim, n, K):
    # moe_layer_forward routes, groups and gathers a batch of T <= 32 tokens
    # over n <= 8 experts in one launch: edge batches (1 token, 32 tokens),
    # K = 1, K = n, fewer than 8 experts, 8x22B's model dimension (with 8
    # experts, a lane's 16-byte slices of W_g come in an odd count), and the
    # most assignments the launch takes (32 x 8)
    cfg = mi.Config("small-route", T=T, dim=dim, hidden=256, n_experts=n, top_k=K,
                    seed=46600 + T * 7 + dim + n)
    assert fused_routes_in_one_launch(cfg)
    check_layer(cfg, 0)


def test_largest_batch_mixtral_dims():
    # T = 65536 at Mixtral dims: T * K * hidden = 1.88e9, just under the 2^31
    # limit of the supported shapes, so byte offsets into x_perm and H run far
    # past 2^31 and every expert's rows are walked in L2-sized blocks; every
    # token is checked (the oracle needs about two minutes)
    cfg = mi.CONFIGS["prefill"].replace(name="max-batch", T=65536, seed=46111)
    check_layer(cfg, 0)
