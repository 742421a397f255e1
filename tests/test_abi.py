"""The C-ABI library loads and exports every entry point include/moe.h declares.

These tests need no GPU: they only load the shared library, read symbols and
exercise host-side argument / shape validation, which returns before any CUDA
call is made.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def build_module():
    import __graft_entry__
    return __graft_entry__._build_module()


@pytest.fixture(scope="module")
def lib():
    path = build_module().build()
    return ctypes.CDLL(path)


def declared_entry_points():
    text = open(HEADER).read()
    return re.findall(r"MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", text)


def test_header_declares_the_boundary_calls():
    names = set(declared_entry_points())
    for required in ("moe_router_topk", "moe_permute", "moe_expert_ffn_grouped",
                     "moe_combine", "moe_layer_forward"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_entry_points()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), name
    from sparse_mixture_experts_46_b300 import _lib
    assert set(_lib.EXPORTS) == set(names)


def test_built_for_sm103a_only():
    assert build_module().ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("dim", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32)]


def test_workspace_size_and_shape_rules(lib):
    lib.moe_workspace_bytes.restype = ctypes.c_size_t
    ok = Shape(4096, 4096, 14336, 8, 2)
    n = lib.moe_workspace_bytes(ctypes.byref(ok))
    R = 4096 * 2
    # at least the grouped activations, hidden activations and expert outputs
    assert n >= R * 4096 * 2 * 2 + R * 14336 * 2
    for bad in [Shape(16, 100, 14336, 8, 2), Shape(16, 4096, 14300, 8, 2),
                Shape(16, 4096, 14336, 33, 2), Shape(16, 4096, 14336, 8, 9),
                Shape(16, 4096, 14336, 8, 0), Shape(-1, 4096, 14336, 8, 2),
                Shape(1 << 20, 4096, 14336, 8, 2), Shape(16, 4096, 14336, 257, 2),
                Shape(16, 4096, 14336, 36, 2), Shape(16, 4096, 14336, 160, 9)]:
        assert lib.moe_workspace_bytes(ctypes.byref(bad)) == 0
    for good in [Shape(16, 4096, 1792, 160, 8), Shape(16, 4096, 14336, 40, 1),
                 Shape(16, 4096, 14336, 256, 8), Shape(16, 4096, 14336, 32, 32)]:
        assert lib.moe_workspace_bytes(ctypes.byref(good)) > 0
    assert lib.moe_workspace_bytes(None) == 0


def test_host_validation_returns_before_any_launch(lib):
    lib.moe_status_string.restype = ctypes.c_char_p
    s = Shape(16, 128, 256, 8, 2)
    vp = ctypes.c_void_p
    # null pointers -> MOE_ERR_INVALID_ARG (1)
    assert lib.moe_router_topk(ctypes.byref(s), None, None, None, None, None, None) == 1
    assert lib.moe_combine(ctypes.byref(s), None, None, None, None, None, None) == 1
    # unsupported shape -> MOE_ERR_UNSUPPORTED_SHAPE (2)
    bad = Shape(16, 100, 256, 8, 2)
    assert lib.moe_router_topk(ctypes.byref(bad), None, None, None, None, None, None) == 2
    # misaligned pointer -> invalid
    assert lib.moe_router_topk(ctypes.byref(s), vp(0x1001), vp(0x2000), vp(0x3000),
                               vp(0x4000), vp(0x5000), None) == 1
    # workspace too small -> MOE_ERR_WORKSPACE_TOO_SMALL (3)
    args = [vp(0x10000)] * 7
    assert lib.moe_permute(ctypes.byref(s), *args, ctypes.c_size_t(4096), None) == 3
    assert lib.moe_status_string(3) == b"MOE_ERR_WORKSPACE_TOO_SMALL"
    assert lib.moe_status_string(5) == b"MOE_ERR_TIMEOUT"


def test_backward_and_stats_shape_rules_and_validation(lib):
    lib.moe_backward_workspace_bytes.restype = ctypes.c_size_t
    vp = ctypes.c_void_p
    # the backward needs dim and hidden multiples of 256
    for bad in (Shape(16, 128, 256, 8, 2), Shape(16, 256, 384, 8, 2), Shape(16, 256, 256, 8, 9)):
        assert lib.moe_backward_workspace_bytes(ctypes.byref(bad)) == 0
    small = lib.moe_backward_workspace_bytes(ctypes.byref(Shape(16, 256, 256, 8, 2)))
    large = lib.moe_backward_workspace_bytes(ctypes.byref(Shape(4096, 256, 256, 8, 2)))
    # the grouped buffers hold at least T*K rows of x_perm, h, [a|g], y_perm, dO, [dA|dG], dx_perm
    assert large > small > 0
    assert large >= 4096 * 2 * (4 * 256 + 5 * 256) * 2
    s = Shape(16, 256, 256, 8, 2)
    p = [vp(0x10000 * (i + 1)) for i in range(11)]
    # null shape / unsupported shape / null pointer / workspace too small: no launch
    assert lib.moe_layer_backward(None, *p, vp(0x200000), ctypes.c_size_t(small), None) == 1
    bad = Shape(16, 128, 256, 8, 2)
    assert lib.moe_layer_backward(ctypes.byref(bad), *p, vp(0x200000), ctypes.c_size_t(small),
                                  None) == 2
    assert lib.moe_layer_backward(ctypes.byref(s), None, *p[1:], vp(0x200000),
                                  ctypes.c_size_t(small), None) == 1
    assert lib.moe_layer_backward(ctypes.byref(s), *p, vp(0x200000), ctypes.c_size_t(small - 1),
                                  None) == 3
    # routing statistics: null outputs and unsupported shapes return before any launch
    assert lib.moe_routing_stats(ctypes.byref(s), vp(0x1000), None, vp(0x2000), None) == 1
    assert lib.moe_routing_stats(ctypes.byref(Shape(16, 256, 256, 8, 9)), vp(0x1000),
                                 vp(0x2000), vp(0x3000), None) == 2
