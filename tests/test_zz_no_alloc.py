"""moe_permute_noalloc: the expert grouping for callers that cannot allocate
device memory (they are handed only input and output buffers by a host
framework with no workspace argument, and may not call cudaMalloc themselves).
It uses the library's fixed device scratch array instead of a caller
workspace; its outputs must equal those of moe_permute, call after call."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from tests.gpu_util import dev_bf16, dev_i32, host_bits, lib

pytestmark = pytest.mark.gpu


def _outputs(cfg):
    R = cfg.T * cfg.top_k
    i32 = dict(dtype=torch.int32, device="cuda")
    return (torch.full((cfg.n_experts + 1,), -3, **i32), torch.full((R,), -3, **i32),
            torch.full((R,), -3, **i32),
            torch.zeros((R, cfg.dim), dtype=torch.bfloat16, device="cuda"))


def _host(outs):
    off, src, slot, xp = outs
    return off.cpu().numpy(), src.cpu().numpy(), slot.cpu().numpy(), host_bits(xp)


def _case(T, n, K, dim, seed):
    cfg = mi.Config("noalloc", T=T, dim=dim, hidden=128, n_experts=n, top_k=K, seed=seed)
    rng = np.random.default_rng(seed)
    ids = np.argsort(rng.random((T, n)), axis=1)[:, :K].astype(np.int32)
    return cfg, dev_bf16(mi.gen_x(cfg)), dev_i32(ids)


def _check_same(cfg, x, ids):
    moe = lib()
    ref = _outputs(cfg)
    moe.moe_permute(cfg, x, ids, *ref, moe.new_workspace(cfg))
    got = _outputs(cfg)
    moe.moe_permute_noalloc(cfg, x, ids, *got)
    torch.cuda.synchronize()
    for a, b in zip(_host(got), _host(ref)):
        assert np.array_equal(a, b)


def test_noalloc_grouping_equals_workspace_grouping_twice():
    # two calls in a row, both above the 8192 assignments that one block or
    # one cluster groups on its own, so both go through the shared scratch
    # tables: the first with the larger table (40 chunks x 16 experts), the
    # second with a smaller one (36 chunks x 8 experts) that must not depend
    # on what the first call left in the scratch
    for T, n, K, dim, seed in [(5000, 16, 2, 256, 11), (4500, 8, 2, 128, 12)]:
        R = T * K
        assert R > 8192
        _check_same(*_case(T, n, K, dim, seed))


def test_noalloc_grouping_at_the_scratch_limit():
    # ceil(T*K / 256) * n == 65536 exactly (256 chunks x 256 experts): the
    # largest table the fixed scratch holds is accepted and matches moe_permute
    cfg, x, ids = _case(8192, 256, 8, 128, 13)
    assert -(-cfg.T * cfg.top_k // 256) * cfg.n_experts == 65536
    _check_same(cfg, x, ids)


@pytest.mark.parametrize("T,n,K", [(2_200_000, 8, 1), (65_537, 256, 1)])
def test_noalloc_rejects_shapes_beyond_its_scratch(T, n, K):
    # the library itself refuses a batch beyond its fixed scratch (here one
    # chunk past it: 257 chunks x 256 experts) before it enqueues anything;
    # called through the C entry point, because the Python binding already
    # refuses these tensors as too small for the shape
    import ctypes
    moe = lib()
    s = moe.make_shape(T=T, dim=128, hidden=128, n_experts=n, top_k=K)
    small = _outputs(mi.Config("s", T=1, dim=128, hidden=128, top_k=1))
    x = torch.zeros((1, 128), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    ptrs = [ctypes.c_void_p(t.data_ptr()) for t in (x, ids, *small)]
    status = moe._lib._LIB.moe_permute_noalloc(ctypes.byref(s), *ptrs, None)
    assert status == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(ValueError, match="holds"):
        moe.moe_permute_noalloc(s, x, ids, *small)
