"""Failure detection without a GPU fault: a bounded device wait that runs out
is reported as MOE_ERR_TIMEOUT, the context stays usable, and bad arguments
are rejected on the host before anything is enqueued."""
import pytest
import torch

import moe_inputs as mi
from tests.gpu_util import lib

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_cleared():
    moe = lib()
    cfg = mi.CONFIGS["tiny"]
    ws = moe.new_workspace(cfg)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    moe.moe_selftest_wait_timeout(ws, 2_000_000)          # 2 ms; nothing ever arrives
    assert moe.moe_check_error(ws) == moe.MOE_ERR_TIMEOUT
    assert moe.moe_check_error(ws) == moe.MOE_OK          # cleared by the check
    # the context is still healthy
    a = torch.ones(1024, device="cuda")
    assert float(a.sum()) == 1024.0


def test_host_side_rejections():
    moe = lib()
    cfg = mi.CONFIGS["tiny"]
    ws = moe.new_workspace(cfg)
    x = torch.zeros((cfg.T, cfg.dim), dtype=torch.bfloat16, device="cuda")
    wg = torch.zeros((cfg.dim, cfg.n_experts), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((cfg.T, 2), dtype=torch.int32, device="cuda")
    gates = torch.zeros((cfg.T, 2), dtype=torch.float32, device="cuda")
    counts = torch.zeros((8,), dtype=torch.int32, device="cuda")
    bad = cfg.replace(dim=100)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_router_topk(bad, x, wg, ids, gates, counts)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED_SHAPE
    small_ws = ws[:4096]
    w = torch.zeros((8, cfg.hidden, cfg.dim), dtype=torch.bfloat16, device="cuda")
    w2 = torch.zeros((8, cfg.dim, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros_like(x)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_layer_forward(cfg, x, wg, w, w, w2, y, small_ws)
    assert e.value.status == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(moe.MoeError) as e:
        moe.moe_layer_forward(cfg, x, wg, w, w, w2, y, ws, ffn_path=7)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
