"""GPU grouped expert FFN (moe_expert_ffn_grouped), both operand layouts,
against the oracle's grouped SwiGLU FFN (fp64, exact mode)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as orc
from tests.gpu_util import assert_bf16_close, dev_bf16, dev_i32, host_bits, lib

pytestmark = pytest.mark.gpu

PATHS = {"gemm": 1, "stream": 2, "pair": 3}


def ffn_case(counts, dim, hidden, seed):
    counts = np.asarray(counts, dtype=np.int64)
    n = len(counts)
    R = int(counts.sum())
    cfg = mi.Config("f", T=R, dim=dim, hidden=hidden, n_experts=n, top_k=1, seed=seed)
    x_perm = mi.gen_x(cfg)                          # [R, dim] grouped rows
    w1, w3, w2 = mi.gen_experts(cfg)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return cfg, x_perm, offsets, w1, w3, w2


def run_ffn(cfg, x_perm, offsets, w1, w3, w2, path):
    moe = lib()
    R = cfg.T * cfg.top_k
    h = torch.full((R, cfg.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
    y_perm = torch.full((R, cfg.dim), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = moe.new_workspace(cfg)
    moe.moe_expert_ffn_grouped(cfg, dev_bf16(x_perm), dev_i32(offsets), dev_bf16(w1),
                               dev_bf16(w3), dev_bf16(w2), h, y_perm, ws, path=PATHS[path])
    status = moe.moe_check_error(ws)
    assert status == moe.MOE_OK, status
    return host_bits(h), host_bits(y_perm)


def diagnose(h_gpu, x_perm, offsets, w1, w3):
    """Describe how a wrong H relates to plausible alternatives (printed on failure)."""
    g = orc.widen_bf16(h_gpu)
    lo, hi = int(offsets[0]), int(offsets[1])
    x = orc.widen_bf16(x_perm[lo:hi])
    cands = {
        "silu(xW1)*xW3": orc.silu(x @ orc.widen_bf16(w1[0]).T) * (x @ orc.widen_bf16(w3[0]).T),
        "xW1": x @ orc.widen_bf16(w1[0]).T,
        "xW3": x @ orc.widen_bf16(w3[0]).T,
        "silu(xW3)*xW1": orc.silu(x @ orc.widen_bf16(w3[0]).T) * (x @ orc.widen_bf16(w1[0]).T),
    }
    out = []
    gg = g[lo:hi]
    for k, v in cands.items():
        m = np.isfinite(gg)
        c = np.corrcoef(gg[m].ravel(), v[m].ravel())[0, 1] if m.sum() > 2 else float("nan")
        out.append("%s corr=%.4f" % (k, c))
    out.append("gpu nan frac=%.3f, gpu[0,:4]=%s ref[0,:4]=%s" % (
        float(np.mean(~np.isfinite(gg))), gg[0, :4], cands["silu(xW1)*xW3"][0, :4]))
    return "; ".join(out)


def check_ffn(counts, dim, hidden, path, seed=1):
    cfg, x_perm, offsets, w1, w3, w2 = ffn_case(counts, dim, hidden, seed)
    h, y_perm = run_ffn(cfg, x_perm, offsets, w1, w3, w2, path)
    ref_y, ref_h = orc.grouped_ffn(x_perm, offsets, w1, w3, w2)
    try:
        assert_bf16_close(h, ref_h, "hidden activations")
    except AssertionError as e:
        raise AssertionError(str(e) + " | " + diagnose(h, x_perm, offsets, w1, w3))
    assert_bf16_close(y_perm, ref_y, "expert outputs")


@pytest.mark.parametrize("path", ["gemm", "stream"])
def test_ffn_single_expert_one_tile(path):
    check_ffn([128], 128, 128, path)


@pytest.mark.parametrize("path", ["gemm", "stream"])
def test_ffn_ragged_groups(path):
    check_ffn([0, 1, 127, 128, 129, 300, 5, 2], 128, 256, path, seed=2)


@pytest.mark.parametrize("path", ["gemm", "stream", "pair"])
def test_ffn_w2_256_wide_tiles(path):
    check_ffn([40, 0, 260, 7], 256, 384, path, seed=3)


@pytest.mark.parametrize("path", ["gemm", "stream"])
def test_ffn_dim_not_multiple_of_256(path):
    check_ffn([33, 200, 1], 384, 128, path, seed=4)


@pytest.mark.parametrize("path", ["gemm", "stream"])
def test_ffn_single_row(path):
    check_ffn([0, 0, 1], 128, 128, path, seed=5)


@pytest.mark.parametrize("counts", [[4] * 8, [0, 5, 0, 11, 0, 0, 16, 0]])
def test_stream_presumed_schedule_prefetch(counts):
    # T = 32 rows over 8 experts with K = 1: (7/8)^32 < 0.05, so each pass of
    # the weight stream requests the first units of the schedule it presumes
    # (every expert touched once) into L2 before its dependency wait; the
    # second case leaves 5 of the 8 experts empty, so the presumption is
    # wrong and only the results show whether the real schedule was followed
    check_ffn(counts, 256, 256, "stream", seed=7)


def test_ffn_paths_agree_bitwise_structure():
    """Both layouts compute the same rows (values within tolerance of each other)."""
    cfg, x_perm, offsets, w1, w3, w2 = ffn_case([17, 33, 0, 64], 256, 256, 6)
    h1, y1 = run_ffn(cfg, x_perm, offsets, w1, w3, w2, "gemm")
    h2, y2 = run_ffn(cfg, x_perm, offsets, w1, w3, w2, "stream")
    ref_y, _ = orc.grouped_ffn(x_perm, offsets, w1, w3, w2)
    assert_bf16_close(y1, ref_y, "gemm")
    assert_bf16_close(y2, ref_y, "stream")
    assert_bf16_close(y1, orc.widen_bf16(y2), "gemm vs stream", atol=2e-2, rtol=2e-2)


# The CTA-pair path (weights on the M side of a two-SM MMA, token tiles of up to
# 256 rows whose MMA N shrinks to the rows left, rounded up to 16) needs dim % 256 == 0.

def test_pair_single_full_tile():
    check_ffn([256], 256, 128, "pair", seed=11)


def test_pair_every_partial_width():
    # last token tiles of 1, 15, 16, 17, 255, 256, 1 (257), 44 (300), 1 (513) rows
    check_ffn([0, 1, 15, 16, 17, 255, 256, 257, 300, 513, 2], 256, 384, "pair", seed=12)


def test_pair_many_tiles_per_pair():
    # 4 x 8 weight tiles per expert for gate/up and 2 for down, several token tiles
    check_ffn([700, 33, 0, 1200], 512, 1024, "pair", seed=13)


def test_pair_long_reduction():
    # down projection over K = 4096: the 6-stage ring wraps many times per tile
    check_ffn([90, 300], 256, 4096, "pair", seed=14)


def test_pair_rejects_dim_not_multiple_of_256():
    moe = lib()
    cfg, x_perm, offsets, w1, w3, w2 = ffn_case([10, 20], 384, 128, 15)
    R = cfg.T
    h = torch.empty((R, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((R, cfg.dim), dtype=torch.bfloat16, device="cuda")
    ws = moe.new_workspace(cfg)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_expert_ffn_grouped(cfg, dev_bf16(x_perm), dev_i32(offsets), dev_bf16(w1),
                                   dev_bf16(w3), dev_bf16(w2), h, y, ws, path=PATHS["pair"])
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED_SHAPE


def test_pair_agrees_with_token_tiles():
    cfg, x_perm, offsets, w1, w3, w2 = ffn_case([129, 0, 511, 64], 512, 256, 16)
    h1, y1 = run_ffn(cfg, x_perm, offsets, w1, w3, w2, "gemm")
    h2, y2 = run_ffn(cfg, x_perm, offsets, w1, w3, w2, "pair")
    ref_y, ref_h = orc.grouped_ffn(x_perm, offsets, w1, w3, w2)
    assert_bf16_close(h2, ref_h, "pair hidden")
    assert_bf16_close(y2, ref_y, "pair out")
    assert_bf16_close(y2, orc.widen_bf16(y1), "pair vs gemm", atol=2e-2, rtol=2e-2)


def test_ffn_many_small_groups_160_experts():
    # fine-grained MoE: 160 experts, most groups tiny or empty
    rng = np.random.default_rng(17)
    counts = rng.integers(0, 9, size=160)
    counts[rng.choice(160, 40, replace=False)] = 0
    counts[3] = 300
    for path in ("pair", "gemm", "stream"):
        check_ffn(counts, 256, 256, path, seed=17)


# The weight stream splits each pass into equal ranges of (tile, K block) units
# over the SMs (stream-K); tiles split between CTAs are summed by the last one.

def test_stream_k_tile_split_over_many_ctas():
    # one expert, 5 rows: the down pass has 2 weight tiles of 32 K blocks each,
    # so every tile is shared by ~74 CTAs; gate/up has 16 tiles of 4 K blocks
    check_ffn([5], 256, 2048, "stream", seed=21)


def test_stream_k_counters_return_to_zero():
    """Three calls on one workspace give identical bits (every split tile's
    arrival counter is back at zero after each call)."""
    moe = lib()
    cfg, x_perm, offsets, w1, w3, w2 = ffn_case([3, 0, 17, 9, 30, 1], 256, 640, 22)
    R = cfg.T
    ws = moe.new_workspace(cfg)
    args = [dev_bf16(x_perm), dev_i32(offsets), dev_bf16(w1), dev_bf16(w3), dev_bf16(w2)]
    outs = []
    for _ in range(3):
        h = torch.full((R, cfg.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
        y = torch.full((R, cfg.dim), float("nan"), dtype=torch.bfloat16, device="cuda")
        moe.moe_expert_ffn_grouped(cfg, args[0], args[1], args[2], args[3], args[4], h, y, ws,
                                   path=PATHS["stream"])
        assert moe.moe_check_error(ws) == moe.MOE_OK
        outs.append((host_bits(h), host_bits(y)))
    ref_y, ref_h = orc.grouped_ffn(x_perm, offsets, w1, w3, w2)
    assert_bf16_close(outs[0][0], ref_h, "hidden activations")
    assert_bf16_close(outs[0][1], ref_y, "expert outputs")
    for h, y in outs[1:]:
        assert np.array_equal(h, outs[0][0]) and np.array_equal(y, outs[0][1])


def test_stream_whole_tile_schedule_beyond_the_stream_k_counters():
    # 256 experts of hidden 8192: a pass can have (R/32 + n) * 64 = 24832 tiles,
    # more than the stream-K arrival counters hold, so the weight stream runs
    # its whole-tile schedule (ragged groups of 0 to 33 rows)
    counts = [[0, 1, 2, 31, 32, 33][e % 6] for e in range(256)]
    check_ffn(counts, 128, 8192, "stream", seed=23)
