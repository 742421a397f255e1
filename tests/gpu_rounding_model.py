"""A model of where the CUDA layer backward stores bf16 intermediates.

NOT the oracle.  The oracle (``oracle/moe_oracle.py``) computes the exact
fp64 gradient and is what parity is judged against; it is pinned on the CPU by
central differences.  This module replays the CUDA path's bf16 storage points
in fp64 so that a second, tighter comparison can separate "the kernel stores a
value in bf16 where it should" (expected, and modelled here) from "the kernel
computes the wrong thing" (caught by both comparisons).  It is a description
of one implementation's rounding, written down from that implementation's
design, and is checked only against the exact oracle
(``tests/test_oracle_pins.py::test_gpu_rounding_model_*``): it must differ
from it by bf16-sized amounts and agree with it where nothing rounds.

Storage points of the CUDA backward (routing held fixed, everything else
accumulated in fp32):
  * the gate/up pre-activations a = W1 x and b = W3 x are saved in bf16; the
    forward's h = SiLU(a) * b is formed from the unrounded fp32 a and b, then
    stored in bf16;
  * the expert outputs o = W2 h are stored in bf16;
  * the upstream gradient scaled by the gate, g_k * dy, is stored in bf16;
  * dA = dH * b * SiLU'(a) and dG = dH * SiLU(a) (from the saved, rounded a
    and b) are stored in bf16;
  * each expert's input-gradient rows dA W1 + dG W3 are stored in bf16 before
    the sum over the K experts of a token.
"""
import numpy as np

from oracle import moe_oracle as orc


def _rnd(v):
    return orc.widen_bf16(orc.round_bf16(v))


def backward_at_gpu_storage_points(x, w_gate, w1, w3, w2, top_k, dy):
    """The layer backward with the CUDA path's bf16 storage points replayed
    (see the module docstring); same outputs as ``orc.moe_layer_backward``."""
    xf, wg = orc._f64(x), orc._f64(w_gate)
    g_up = orc._f64(dy)
    ids, gates, _ = orc.router(xf, wg, top_k)
    T, dim = xf.shape
    n = np.asarray(w1).shape[0]
    dx = np.zeros_like(xf)
    dwg = np.zeros_like(wg)
    dw1 = np.zeros(np.asarray(w1).shape)
    dw3 = np.zeros(np.asarray(w3).shape)
    dw2 = np.zeros(np.asarray(w2).shape)
    dgate = np.zeros((T, top_k))
    for e in range(n):
        tok, slot = np.nonzero(ids == e)
        if len(tok) == 0:
            continue
        W1e, W3e, W2e = orc._f64(w1[e]), orc._f64(w3[e]), orc._f64(w2[e])
        xe = xf[tok]
        a_x = xe @ W1e.T
        b_x = xe @ W3e.T
        h = _rnd(orc.silu(a_x) * b_x)
        a, b = _rnd(a_x), _rnd(b_x)
        s = orc.silu(a)
        o = _rnd(h @ W2e.T)
        do = _rnd(gates[tok, slot][:, None] * g_up[tok])
        dgate[tok, slot] = np.sum(g_up[tok] * o, axis=1)
        dh = do @ W2e
        da = _rnd(dh * b * orc.silu_grad(a))
        db = _rnd(dh * s)
        dw2[e] += do.T @ h
        dw1[e] += da.T @ xe
        dw3[e] += db.T @ xe
        np.add.at(dx, tok, _rnd(da @ W1e + db @ W3e))
    dl_sel = gates * (dgate - np.sum(gates * dgate, axis=1, keepdims=True))
    dl = np.zeros((T, n))
    np.put_along_axis(dl, ids, dl_sel, axis=1)
    dwg += xf.T @ dl
    dx += dl @ wg.T
    return dict(dx=dx, dwg=dwg, dw1=dw1, dw3=dw3, dw2=dw2)
