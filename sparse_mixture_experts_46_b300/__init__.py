"""B300 (sm_103a) Mixtral sparse mixture-of-experts layer forward.

The computation runs entirely in the CUDA library ``libmoe_b300.so``
(``csrc/``, C ABI in ``include/moe.h``); this package only marshals torch
tensors into its entry points.  ``MoELayer`` is a convenience holder of one
layer's device weights and workspace.
"""
from __future__ import annotations

import torch

from ._lib import (  # noqa: F401
    EXPORTS, LIB_PATH, MOE_ERR_CUDA, MOE_ERR_INVALID_ARG, MOE_ERR_TIMEOUT,
    MOE_ERR_UNSUPPORTED_SHAPE, MOE_ERR_WORKSPACE_TOO_SMALL, MOE_FFN_AUTO, MOE_FFN_GROUPED_GEMM,
    MOE_FFN_PAIR_GEMM, MOE_FFN_WEIGHT_STREAM, MOE_OK, MoeError, MoeShape, make_shape, moe_check_error,
    moe_combine, moe_expert_ffn_grouped, moe_layer_forward, moe_permute, moe_permute_noalloc,
    moe_router_topk, moe_routing_stats, moe_backward_workspace_bytes, moe_layer_backward,
    new_backward_workspace,
    moe_selftest_wait_timeout, moe_workspace_bytes, moe_workspace_init, new_workspace)


class MoELayer:
    """One sparse MoE layer resident on the GPU.

    w_gate [dim, n], w1/w3 [n, hidden, dim], w2 [n, dim, hidden]: bf16 tensors
    on the device.  ``forward(x)`` returns y [T, dim] bf16 on the current
    stream; the workspace grows to the largest T seen.
    """

    def __init__(self, w_gate, w1, w3, w2, top_k: int = 2):
        self.w_gate, self.w1, self.w3, self.w2 = w_gate, w1, w3, w2
        self.dim, self.n_experts = w_gate.shape
        self.hidden = w1.shape[1]
        self.top_k = top_k
        self._ws = None
        self._ws_T = -1

    def shape(self, T: int) -> MoeShape:
        return make_shape(T, self.dim, self.hidden, self.n_experts, self.top_k)

    def workspace(self, T: int) -> torch.Tensor:
        if self._ws is None or T > self._ws_T:
            self._ws = new_workspace(self.shape(T), device=self.w_gate.device)
            self._ws_T = T
        return self._ws

    def forward(self, x, y=None, ids=None, gates=None, rmsnorm_eps=None, residual=None,
                ffn_path=MOE_FFN_AUTO, stream=None):
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.dim), dtype=x.dtype, device=x.device)
        ws = self.workspace(T)
        moe_layer_forward(self.shape(T), x, self.w_gate, self.w1, self.w3, self.w2, y, ws,
                          ids=ids, gates=gates, rmsnorm_eps=rmsnorm_eps, residual=residual,
                          ffn_path=ffn_path, stream=stream)
        return y

    __call__ = forward
