"""ctypes binding of libmoe_b300.so (include/moe.h): argument marshalling only.

Every function here has the name of the C entry point it calls, takes torch
tensors that already live on the GPU, checks dtype / device / contiguity,
passes ``data_ptr()`` and the current CUDA stream, and raises ``MoeError`` on a
non-OK status.  No computation happens in Python; if the shared library is
missing, importing this module fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_b300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_WORKSPACE_TOO_SMALL = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5

MOE_FFN_AUTO = 0
MOE_FFN_GROUPED_GEMM = 1
MOE_FFN_WEIGHT_STREAM = 2
MOE_FFN_PAIR_GEMM = 3

# Every symbol include/moe.h declares.
EXPORTS = (
    "moe_status_string", "moe_workspace_bytes", "moe_workspace_init", "moe_router_topk",
    "moe_permute", "moe_expert_ffn_grouped", "moe_combine", "moe_layer_forward",
    "moe_check_error", "moe_selftest_wait_timeout", "moe_permute_noalloc", "moe_routing_stats",
    "moe_backward_workspace_bytes", "moe_layer_backward",
)


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("dim", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32)]


class MoeLayerOpts(ctypes.Structure):
    _fields_ = [("use_rmsnorm", ctypes.c_int32), ("rmsnorm_eps", ctypes.c_float),
                ("residual", ctypes.c_void_p), ("ffn_path", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s" % (where, _status_name(status)))


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "libmoe_b300.so is not built (%s); run `python -m "
            "sparse_mixture_experts_46_b300.build` or __graft_entry__.build()" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
    sp = ctypes.POINTER(MoeShape)
    sig = {
        "moe_status_string": (ctypes.c_char_p, [i32]),
        "moe_workspace_bytes": (sz, [sp]),
        "moe_workspace_init": (i32, [vp, sz, vp]),
        "moe_router_topk": (i32, [sp, vp, vp, vp, vp, vp, vp]),
        "moe_permute": (i32, [sp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "moe_expert_ffn_grouped": (i32, [sp, vp, vp, vp, vp, vp, vp, vp, i32, vp, sz, vp]),
        "moe_combine": (i32, [sp, vp, vp, vp, vp, vp, vp]),
        "moe_layer_forward": (i32, [sp, ctypes.POINTER(MoeLayerOpts), vp, vp, vp, vp, vp, vp, vp,
                                    vp, vp, sz, vp]),
        "moe_check_error": (i32, [vp, vp]),
        "moe_selftest_wait_timeout": (i32, [vp, sz, ctypes.c_uint64, vp]),
        "moe_permute_noalloc": (i32, [sp, vp, vp, vp, vp, vp, vp, vp]),
        "moe_routing_stats": (i32, [sp, vp, vp, vp, vp]),
        "moe_backward_workspace_bytes": (sz, [sp]),
        "moe_layer_backward": (i32, [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_LIB = _load()


def _status_name(status: int) -> str:
    return _LIB.moe_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)


def make_shape(T, dim, hidden, n_experts, top_k) -> MoeShape:
    return MoeShape(int(T), int(dim), int(hidden), int(n_experts), int(top_k))


def _shape(shape) -> MoeShape:
    if isinstance(shape, MoeShape):
        return shape
    if hasattr(shape, "T") and hasattr(shape, "dim"):
        return make_shape(shape.T, shape.dim, shape.hidden, shape.n_experts, shape.top_k)
    return make_shape(*shape)


_BF16 = (torch.bfloat16, torch.uint16, torch.int16)


def _need(*checks):
    """Element counts, checked for every argument of a call before any pointer
    is taken: each (tensor or None, elements the shape implies, name).  A
    shorter tensor would let a kernel read or write past it."""
    for t, numel, name in checks:
        if isinstance(t, torch.Tensor) and t.numel() < numel:
            raise ValueError("%s holds %d elements; the shape needs %d"
                             % (name, t.numel(), numel))


def _ptr(t, dtypes=None, name="tensor", nullable=False):
    """Device pointer of a tensor after the checks the C ABI cannot make (type,
    device, layout, dtype; element counts are _need's)."""
    if t is None:
        if nullable:
            return None
        raise ValueError("%s is required" % name)
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


_I32 = (torch.int32,)
_F32 = (torch.float32,)


def _sizes(s):
    """Element counts of every array of the boundary for shape s."""
    T, d, h, n, K = s.T, s.dim, s.hidden, s.n_experts, s.top_k
    R = T * K
    return dict(x=T * d, wg=d * n, w=n * h * d, tk=R, n=n, off=n + 1, xp=R * d, hp=R * h)


def moe_workspace_bytes(shape) -> int:
    s = _shape(shape)
    n = _LIB.moe_workspace_bytes(ctypes.byref(s))
    if n == 0:
        raise MoeError(MOE_ERR_UNSUPPORTED_SHAPE, "moe_workspace_bytes")
    return int(n)


def moe_workspace_init(ws, stream=None) -> None:
    _check(_LIB.moe_workspace_init(_ptr(ws, name="ws"), ws.numel() * ws.element_size(),
                                   _stream(stream)), "moe_workspace_init")


def new_workspace(shape, device=None, stream=None) -> torch.Tensor:
    """Allocate (through torch) and initialise a workspace for ``shape``."""
    ws = torch.empty(moe_workspace_bytes(shape), dtype=torch.uint8,
                     device=device or torch.device("cuda"))
    moe_workspace_init(ws, stream)
    return ws


def moe_router_topk(shape, x, w_gate, ids, gates, counts, stream=None) -> None:
    s = _shape(shape)
    z = _sizes(s)
    _need((x, z["x"], "x"),
          (w_gate, z["wg"], "w_gate"),
          (ids, z["tk"], "ids"),
          (gates, z["tk"], "gates"),
          (counts, z["n"], "counts"))
    _check(_LIB.moe_router_topk(ctypes.byref(s), _ptr(x, _BF16, "x"),
                                _ptr(w_gate, _BF16, "w_gate"),
                                _ptr(ids, _I32, "ids"),
                                _ptr(gates, _F32, "gates"),
                                _ptr(counts, _I32, "counts"),
                                _stream(stream)), "moe_router_topk")


def moe_permute(shape, x, ids, offsets, perm_src, slot_row, x_perm, ws, stream=None) -> None:
    s = _shape(shape)
    z = _sizes(s)
    _need((x, z["x"], "x"),
          (ids, z["tk"], "ids"),
          (offsets, z["off"], "offsets"),
          (perm_src, z["tk"], "perm_src"),
          (slot_row, z["tk"], "slot_row"),
          (x_perm, z["xp"], "x_perm"))
    _check(_LIB.moe_permute(ctypes.byref(s), _ptr(x, _BF16, "x"),
                            _ptr(ids, _I32, "ids"),
                            _ptr(offsets, _I32, "offsets"),
                            _ptr(perm_src, _I32, "perm_src"),
                            _ptr(slot_row, _I32, "slot_row"),
                            _ptr(x_perm, _BF16, "x_perm"),
                            _ptr(ws, name="ws"), ws.numel() * ws.element_size(),
                            _stream(stream)), "moe_permute")


def moe_expert_ffn_grouped(shape, x_perm, offsets, w1, w3, w2, h, y_perm, ws,
                           path=MOE_FFN_AUTO, stream=None) -> None:
    s = _shape(shape)
    z = _sizes(s)
    _need((x_perm, z["xp"], "x_perm"),
          (offsets, z["off"], "offsets"),
          (w1, z["w"], "w1"),
          (w3, z["w"], "w3"),
          (w2, z["w"], "w2"),
          (h, z["hp"], "h"),
          (y_perm, z["xp"], "y_perm"))
    _check(_LIB.moe_expert_ffn_grouped(
        ctypes.byref(s), _ptr(x_perm, _BF16, "x_perm"),
        _ptr(offsets, _I32, "offsets"),
        _ptr(w1, _BF16, "w1"), _ptr(w3, _BF16, "w3"),
        _ptr(w2, _BF16, "w2"), _ptr(h, _BF16, "h"),
        _ptr(y_perm, _BF16, "y_perm"), int(path), _ptr(ws, name="ws"),
        ws.numel() * ws.element_size(), _stream(stream)), "moe_expert_ffn_grouped")


def moe_combine(shape, y_perm, slot_row, gates, y, residual=None, stream=None) -> None:
    s = _shape(shape)
    z = _sizes(s)
    _need((y_perm, z["xp"], "y_perm"),
          (slot_row, z["tk"], "slot_row"),
          (gates, z["tk"], "gates"),
          (residual, z["x"], "residual"),
          (y, z["x"], "y"))
    _check(_LIB.moe_combine(ctypes.byref(s), _ptr(y_perm, _BF16, "y_perm"),
                            _ptr(slot_row, _I32, "slot_row"),
                            _ptr(gates, _F32, "gates"),
                            _ptr(residual, _BF16, "residual", nullable=True),
                            _ptr(y, _BF16, "y"), _stream(stream)), "moe_combine")


def moe_backward_workspace_bytes(shape) -> int:
    s = _shape(shape)
    n = _LIB.moe_backward_workspace_bytes(ctypes.byref(s))
    if n == 0:
        raise MoeError(MOE_ERR_UNSUPPORTED_SHAPE, "moe_backward_workspace_bytes")
    return int(n)


def new_backward_workspace(shape, device=None, stream=None) -> torch.Tensor:
    """Allocate (through torch) and initialise a workspace for moe_layer_backward."""
    ws = torch.empty(moe_backward_workspace_bytes(shape), dtype=torch.uint8,
                     device=device or torch.device("cuda"))
    moe_workspace_init(ws, stream)
    return ws


def moe_layer_backward(shape, x, w_gate, w1, w3, w2, dy, dx, dw_gate, dw1, dw3, dw2, ws,
                       stream=None) -> None:
    s = _shape(shape)
    z = _sizes(s)
    _need((x, z["x"], "x"),
          (w_gate, z["wg"], "w_gate"),
          (w1, z["w"], "w1"),
          (w3, z["w"], "w3"),
          (w2, z["w"], "w2"),
          (dy, z["x"], "dy"),
          (dx, z["x"], "dx"),
          (dw_gate, z["wg"], "dw_gate"),
          (dw1, z["w"], "dw1"),
          (dw3, z["w"], "dw3"),
          (dw2, z["w"], "dw2"))
    _check(_LIB.moe_layer_backward(
        ctypes.byref(s), _ptr(x, _BF16, "x"),
        _ptr(w_gate, _BF16, "w_gate"), _ptr(w1, _BF16, "w1"),
        _ptr(w3, _BF16, "w3"), _ptr(w2, _BF16, "w2"),
        _ptr(dy, _BF16, "dy"), _ptr(dx, _BF16, "dx"),
        _ptr(dw_gate, _F32, "dw_gate"), _ptr(dw1, _F32, "dw1"),
        _ptr(dw3, _F32, "dw3"), _ptr(dw2, _F32, "dw2"),
        _ptr(ws, name="ws"), ws.numel() * ws.element_size(), _stream(stream)),
        "moe_layer_backward")


def moe_routing_stats(shape, ids, slot_counts, repeats, stream=None) -> None:
    s = _shape(shape)
    z = _sizes(s)
    _need((ids, z["tk"], "ids"),
          (slot_counts, s.top_k * s.n_experts, "slot_counts"),
          (repeats, 2, "repeats"))
    _check(_LIB.moe_routing_stats(ctypes.byref(s), _ptr(ids, _I32, "ids"),
                                  _ptr(slot_counts, _I32, "slot_counts"),
                                  _ptr(repeats, _I32, "repeats"), _stream(stream)),
           "moe_routing_stats")


def moe_layer_forward(shape, x, w_gate, w1, w3, w2, y, ws, ids=None, gates=None,
                      rmsnorm_eps=None, residual=None, ffn_path=MOE_FFN_AUTO,
                      stream=None) -> None:
    s = _shape(shape)
    z = _sizes(s)
    _need((residual, z["x"], "residual"),
          (x, z["x"], "x"),
          (w_gate, z["wg"], "w_gate"),
          (w1, z["w"], "w1"),
          (w3, z["w"], "w3"),
          (w2, z["w"], "w2"),
          (y, z["x"], "y"),
          (ids, z["tk"], "ids"),
          (gates, z["tk"], "gates"))
    opts = MoeLayerOpts(1 if rmsnorm_eps is not None else 0,
                        float(rmsnorm_eps) if rmsnorm_eps is not None else 0.0,
                        _ptr(residual, _BF16, "residual", nullable=True),
                        int(ffn_path))
    _check(_LIB.moe_layer_forward(
        ctypes.byref(s), ctypes.byref(opts), _ptr(x, _BF16, "x"),
        _ptr(w_gate, _BF16, "w_gate"), _ptr(w1, _BF16, "w1"),
        _ptr(w3, _BF16, "w3"), _ptr(w2, _BF16, "w2"),
        _ptr(y, _BF16, "y"), _ptr(ids, _I32, "ids", nullable=True),
        _ptr(gates, _F32, "gates", nullable=True), _ptr(ws, name="ws"),
        ws.numel() * ws.element_size(), _stream(stream)), "moe_layer_forward")


def moe_check_error(ws, stream=None) -> int:
    """Synchronise, read and clear the workspace error word; returns the status."""
    return int(_LIB.moe_check_error(_ptr(ws, name="ws"), _stream(stream)))


def moe_selftest_wait_timeout(ws, limit_ns: int, stream=None) -> None:
    _check(_LIB.moe_selftest_wait_timeout(_ptr(ws, name="ws"), ws.numel() * ws.element_size(),
                                          int(limit_ns), _stream(stream)),
           "moe_selftest_wait_timeout")


def moe_permute_noalloc(shape, x, ids, offsets, perm_src, slot_row, x_perm, stream=None) -> None:
    """moe_permute for callers that cannot allocate a workspace: the library's
    own fixed device scratch is used instead (see include/moe.h)."""
    s = _shape(shape)
    z = _sizes(s)
    _need((x, z["x"], "x"),
          (ids, z["tk"], "ids"),
          (offsets, z["off"], "offsets"),
          (perm_src, z["tk"], "perm_src"),
          (slot_row, z["tk"], "slot_row"),
          (x_perm, z["xp"], "x_perm"))
    _check(_LIB.moe_permute_noalloc(ctypes.byref(s), _ptr(x, _BF16, "x"),
                                    _ptr(ids, _I32, "ids"),
                                    _ptr(offsets, _I32, "offsets"),
                                    _ptr(perm_src, _I32, "perm_src"),
                                    _ptr(slot_row, _I32, "slot_row"),
                                    _ptr(x_perm, _BF16, "x_perm"),
                                    _stream(stream)),
           "moe_permute_noalloc")
