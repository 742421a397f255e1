"""Helpers of the GPU parity tests: device transfer of bf16 bit arrays and the
element-wise acceptance criterion |gpu - ref| <= atol + rtol * |ref|."""
import numpy as np
import torch

from oracle import moe_oracle as orc

ATOL = 1e-2   # bf16 outputs: |gpu - oracle| <= 1e-2 + 1e-2 * |oracle|
RTOL = 1e-2


def lib():
    """The CUDA binding; raises if the shared library is missing."""
    import sparse_mixture_experts_46_b300 as moe
    return moe


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """bf16 bit array (numpy uint16) -> contiguous torch.bfloat16 CUDA tensor."""
    a = np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(a).cuda().view(torch.bfloat16)


def dev_i32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    """torch.bfloat16 tensor -> numpy uint16 bit array."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def empty_bf16(*shape) -> torch.Tensor:
    return torch.empty(shape, dtype=torch.bfloat16, device="cuda")


def assert_bf16_close(gpu_bits, ref, what="", atol=ATOL, rtol=RTOL):
    """Every element: |gpu - ref| <= atol + rtol * |ref| (ref in float64)."""
    g = orc.widen_bf16(gpu_bits)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    err = np.abs(g - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any() or not np.all(np.isfinite(g)):
        idx = np.argwhere(bad | ~np.isfinite(g))[:5]
        raise AssertionError("%s: %d/%d elements out of tolerance; max err %.3g; first %s: gpu %s ref %s"
                             % (what, int(bad.sum()), bad.size, float(np.nanmax(err)),
                                idx.tolist(), [float(g[tuple(i)]) for i in idx],
                                [float(ref[tuple(i)]) for i in idx]))
    return float(err.max()) if err.size else 0.0


# ------------------------------------------------------------- canaries ---
# Out-of-bounds writes cannot be caught by a sanitizer on the test machines,
# so outputs are handed to the library as the head of a larger buffer whose
# tail holds a sentinel; a write past the end of an output changes the tail.

CANARY_ROWS = 3
_SENTINEL = {torch.bfloat16: -12345.0, torch.float32: -1.2345e30, torch.int32: -0x5A5A5A5B,
             torch.uint8: 0xA5}


class Guarded:
    """``view`` (shape ``shape``) is the head of ``full``; the trailing
    CANARY_ROWS rows of ``full`` (``tail`` elements for a 1-D buffer, by
    default CANARY_ROWS * 64) hold a sentinel that ``check()`` requires
    unchanged.  ``fill`` (optional) is written over the head."""

    def __init__(self, shape, dtype, fill=None, tail=None):
        shape = tuple(shape)
        if tail is None:
            tail = CANARY_ROWS if len(shape) > 1 else CANARY_ROWS * 64
        self.rows = shape[0]
        self.full = torch.full((shape[0] + tail, *shape[1:]), _SENTINEL[dtype], dtype=dtype,
                               device="cuda")
        self.view = self.full[:shape[0]]
        if fill is not None:
            self.view.fill_(fill)
        self.tail_ref = self.full[shape[0]:].clone()

    def check(self, what=""):
        tail = self.full[self.rows:].contiguous().view(torch.uint8)
        ref = self.tail_ref.contiguous().view(torch.uint8)
        assert torch.equal(tail, ref), "%s: write past the end of the buffer (canary changed)" % what


def guarded_workspace(moe, cfg, backward=False):
    """A workspace of exactly the size the library asks for, followed by 4 KB
    of sentinel bytes, initialised; returns (ws, Guarded)."""
    nbytes = moe.moe_backward_workspace_bytes(cfg) if backward else moe.moe_workspace_bytes(cfg)
    g = Guarded((nbytes,), torch.uint8, tail=4096)
    moe.moe_workspace_init(g.view)
    return g.view, g
