"""GPU grouped expert FFN (moe_expert_ffn_grouped), both operand layouts,
against the oracle's grouped SwiGLU FFN (fp64, exact mode)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as orc
from tests.gpu_util import assert_bf16_close, dev_bf16, dev_i32, host_bits, lib

pytestmark = pytest.mark.gpu

PATHS = {"gemm": 1, "stream": 2}


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


@pytest.mark.parametrize("path", ["gemm", "stream"])
def test_ffn_w2_256_wide_tiles(path):
    check_ffn([40, 0, 260, 7], 256, 384, path, seed=3)


@pytest.mark.parametrize("path", ["gemm", "stream"])
def test_ffn_dim_not_multiple_of_256(path):
    check_ffn([33, 200, 1], 384, 128, path, seed=4)


@pytest.mark.parametrize("path", ["gemm", "stream"])
def test_ffn_single_row(path):
    check_ffn([0, 0, 1], 128, 128, path, seed=5)


def test_ffn_paths_agree_bitwise_structure():
    """Both layouts compute the same rows (values within tolerance of each other)."""
    cfg, x_perm, offsets, w1, w3, w2 = ffn_case([17, 33, 0, 64], 256, 256, 6)
    h1, y1 = run_ffn(cfg, x_perm, offsets, w1, w3, w2, "gemm")
    h2, y2 = run_ffn(cfg, x_perm, offsets, w1, w3, w2, "stream")
    ref_y, _ = orc.grouped_ffn(x_perm, offsets, w1, w3, w2)
    assert_bf16_close(y1, ref_y, "gemm")
    assert_bf16_close(y2, ref_y, "stream")
    assert_bf16_close(y1, orc.widen_bf16(y2), "gemm vs stream", atol=2e-2, rtol=2e-2)
