"""Test-side input shaping: the router-gap filter.

Routing is compared bit-exactly only where it is decided by a margin far above
fp32 rounding.  Every token whose fp64 oracle logits have a gap below
``MIN_GAP_SELECT`` between the K-th and (K+1)-th largest logit (the selection
boundary), or below ``MIN_GAP_ORDER`` between two consecutive selected logits
(the slot order), is redrawn from the next x stream attempt of the input
generator, up to ``MAX_ATTEMPTS`` times.  This uses the oracle and therefore
lives with the tests, not with the shared input generator.
"""
import numpy as np

import moe_inputs as mi
from oracle import moe_oracle as orc

MIN_GAP_SELECT = 1e-2
MIN_GAP_ORDER = 1e-4
MAX_ATTEMPTS = 64


def ambiguous_tokens(x_bits, wg_bits, top_k):
    """Boolean mask of tokens whose routing is decided by less than the margins."""
    logits = orc.router_logits(x_bits, wg_bits)
    srt = -np.sort(-logits, axis=1)
    n = srt.shape[1]
    bad = np.zeros(srt.shape[0], dtype=bool)
    if top_k < n:
        bad |= (srt[:, top_k - 1] - srt[:, top_k]) < MIN_GAP_SELECT
    for k in range(top_k - 1):
        bad |= (srt[:, k] - srt[:, k + 1]) < MIN_GAP_ORDER
    return bad


def filter_x(cfg, x_bits, wg_bits, shift=None):
    """Redraw ambiguous tokens in place; returns the number of redrawn rows."""
    redrawn = 0
    for attempt in range(1, MAX_ATTEMPTS + 1):
        bad = ambiguous_tokens(x_bits, wg_bits, cfg.top_k)
        if not bad.any():
            return redrawn
        rows = np.nonzero(bad)[0]
        x_bits[rows] = mi.gen_x_rows(cfg, rows, attempt, shift)
        redrawn += len(rows)
    raise RuntimeError("gap filter did not converge")


def filtered_layer(cfg, layer=0, experts=True):
    """Generator inputs of ``cfg`` with the gap filter applied to x."""
    L = mi.make_layer(cfg, layer, experts)
    L.redrawn = filter_x(cfg, L.x, L.wg, L.shift)
    return L
