"""The library on CUDA streams and inside CUDA graphs: moe_layer_forward
captured once into a graph and replayed on new inputs, and two layers running
concurrently on two streams, each with its own workspace.  Every kernel sums
in a fixed order, so both must reproduce the eager single-stream outputs bit
for bit; the eager outputs themselves are checked against the oracle by the
layer tests."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from tests.gpu_util import dev_bf16, host_bits, lib

pytestmark = pytest.mark.gpu

# a decode-sized batch (one-launch routing, weight stream), a batch on the
# CTA-pair path, and one with RMSNorm and a residual (router + grouping kernels)
SHAPES = {
    "decode": dict(T=16, dim=1024, hidden=1024, n_experts=8, top_k=2),
    "pair": dict(T=600, dim=512, hidden=768, n_experts=8, top_k=2),
    "norm_residual": dict(T=96, dim=256, hidden=512, n_experts=8, top_k=2),
}


class Layer:
    def __init__(self, name, seed):
        self.cfg = mi.Config(name, seed=seed, **SHAPES[name])
        L = mi.make_layer(self.cfg)
        self.wg, self.w1, self.w3, self.w2 = (dev_bf16(a) for a in (L.wg, L.w1, L.w3, L.w2))
        self.norm = name == "norm_residual"
        self.moe = lib()

    def inputs(self, seed):
        return dev_bf16(mi.gen_x(self.cfg.replace(seed=seed)))

    def forward(self, x, y, ws, stream=None):
        kw = dict(rmsnorm_eps=1e-5, residual=x) if self.norm else {}
        self.moe.moe_layer_forward(self.cfg, x, self.wg, self.w1, self.w3, self.w2, y, ws,
                                   stream=stream, **kw)

    def eager(self, x):
        y = torch.empty_like(x)
        ws = self.moe.new_workspace(self.cfg)
        self.forward(x, y, ws)
        assert self.moe.moe_check_error(ws) == self.moe.MOE_OK
        return host_bits(y)


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_layer_forward_replays_from_a_cuda_graph(name):
    layer = Layer(name, seed=47000 + len(name))
    xs = [layer.inputs(47100 + i) for i in range(3)]
    want = [layer.eager(x) for x in xs]
    moe = layer.moe
    static_x = torch.empty_like(xs[0])
    static_y = torch.empty_like(xs[0])
    ws = moe.new_workspace(layer.cfg)
    # warm-up on a side stream (host-side caches: tensor-map encoder, grids)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        static_x.copy_(xs[0])
        layer.forward(static_x, static_y, ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(static_x, static_y, ws)
    for x, ref in list(zip(xs, want)) + list(zip(xs[::-1], want[::-1])):
        static_x.copy_(x)
        static_y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(static_y), ref)
    assert moe.moe_check_error(ws) == moe.MOE_OK


def test_two_layers_on_two_streams():
    a, b = Layer("decode", seed=47200), Layer("pair", seed=47201)
    xa = [a.inputs(47300 + i) for i in range(4)]
    xb = [b.inputs(47400 + i) for i in range(4)]
    want_a = [a.eager(x) for x in xa]
    want_b = [b.eager(x) for x in xb]
    moe = a.moe
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    wsa, wsb = moe.new_workspace(a.cfg), moe.new_workspace(b.cfg)
    ya = [torch.full_like(x, float("nan")) for x in xa]
    yb = [torch.full_like(x, float("nan")) for x in xb]
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    for i in range(4):  # both streams busy at once, each reusing its workspace
        a.forward(xa[i], ya[i], wsa, stream=sa)
        b.forward(xb[i], yb[i], wsb, stream=sb)
    torch.cuda.synchronize()
    for i in range(4):
        assert np.array_equal(host_bits(ya[i]), want_a[i]), i
        assert np.array_equal(host_bits(yb[i]), want_b[i]), i
    assert moe.moe_check_error(wsa, stream=sa) == moe.MOE_OK
    assert moe.moe_check_error(wsb, stream=sb) == moe.MOE_OK
