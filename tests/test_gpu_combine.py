"""GPU gated combine (moe_combine) against the oracle's weighted sum."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as orc
from tests.gpu_util import assert_bf16_close, dev_bf16, dev_f32, dev_i32, host_bits, lib

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,dim,K,residual", [(1, 128, 2, False), (129, 256, 2, False),
                                               (1000, 4096, 2, True), (50, 384, 8, False),
                                               (64, 128, 1, True)])
def test_combine_matches_oracle(T, dim, K, residual):
    moe = lib()
    rng = np.random.default_rng(T + dim)
    cfg = mi.Config("c", T=T, dim=dim, hidden=128, n_experts=8, top_k=K, seed=T)
    R = T * K
    y_perm = mi.f32_to_bf16(rng.standard_normal((R, dim)).astype(np.float32))
    slot_row = rng.permutation(R).astype(np.int32)
    g = rng.random((T, K)) + 0.01
    gates = (g / g.sum(1, keepdims=True)).astype(np.float32)
    res = mi.gen_x(cfg) if residual else None
    y = torch.empty((T, dim), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(cfg, dev_bf16(y_perm), dev_i32(slot_row), dev_f32(gates), y,
                    residual=dev_bf16(res) if residual else None)
    torch.cuda.synchronize()
    ref = orc.combine(y_perm, slot_row, gates.astype(np.float64), res)
    assert_bf16_close(host_bits(y), ref, "combine")
