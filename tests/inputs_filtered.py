"""Test-side input shaping and routing comparison.

Which experts a token selects is compared bit-exactly only where the selection
is decided by a margin far above fp32 rounding: every token whose fp64 oracle
logits have a gap below ``MIN_GAP_SELECT`` between the K-th and (K+1)-th
largest logit (the selection boundary) is redrawn from the next x stream
attempt of the input generator, up to ``MAX_ATTEMPTS`` times.

The ORDER of the selected experts (slot 0 holds the larger logit) is decided
only where consecutive selected logits differ by at least ``MIN_GAP_ORDER``
(about 100x the fp32 accumulation error of a logit).  Tokens below that margin
are kept, not redrawn: their ids are compared as a set, and their gates and
grouped rows after aligning the GPU's slots to the oracle's by expert id
(``align_slots``).  This uses the oracle and therefore lives with the tests,
not with the shared input generator.
"""
import numpy as np

import moe_inputs as mi
from oracle import moe_oracle as orc

MIN_GAP_SELECT = 1e-2
MIN_GAP_ORDER = 1e-4
MAX_ATTEMPTS = 64


def _sorted_logits(x_bits, wg_bits):
    return -np.sort(-orc.router_logits(x_bits, wg_bits), axis=1)


def ambiguous_tokens(x_bits, wg_bits, top_k):
    """Boolean mask of tokens whose selected SET is decided by less than MIN_GAP_SELECT."""
    srt = _sorted_logits(x_bits, wg_bits)
    if top_k >= srt.shape[1]:
        return np.zeros(srt.shape[0], dtype=bool)
    return (srt[:, top_k - 1] - srt[:, top_k]) < MIN_GAP_SELECT


def order_decided(x_bits, wg_bits, top_k):
    """Boolean mask of tokens whose slot ORDER is decided by at least MIN_GAP_ORDER."""
    srt = _sorted_logits(x_bits, wg_bits)
    ok = np.ones(srt.shape[0], dtype=bool)
    for k in range(top_k - 1):
        ok &= (srt[:, k] - srt[:, k + 1]) >= MIN_GAP_ORDER
    return ok


def filter_x(cfg, x_bits, wg_bits, shift=None):
    """Redraw tokens with an undecided selection in place; returns the number of redrawn rows."""
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


def align_slots(got_ids, ref_ids, decided):
    """Per-token slot permutation p with got_ids[t, p[t, k]] == ref_ids[t, k].

    Raises AssertionError when a token's selected SET differs from the
    oracle's, or when a token whose order is decided (``decided[t]``) has its
    slots in another order.  Returns p ([T, K] int) for aligning the GPU's
    per-slot arrays (gates, slot_row) to the oracle's slot order.
    """
    got_ids = np.asarray(got_ids)
    ref_ids = np.asarray(ref_ids)
    assert got_ids.shape == ref_ids.shape, (got_ids.shape, ref_ids.shape)
    T, K = ref_ids.shape
    same_set = np.array_equal(np.sort(got_ids, axis=1), np.sort(ref_ids, axis=1))
    if not same_set:
        bad = np.nonzero(np.any(np.sort(got_ids, axis=1) != np.sort(ref_ids, axis=1), axis=1))[0]
        raise AssertionError("selected experts differ on %d tokens, first %s: gpu %s ref %s"
                             % (len(bad), bad[:5].tolist(), got_ids[bad[:5]].tolist(),
                                ref_ids[bad[:5]].tolist()))
    exact = np.all(got_ids == ref_ids, axis=1)
    wrong_order = np.nonzero(np.asarray(decided) & ~exact)[0]
    assert len(wrong_order) == 0, ("slot order differs on decided tokens", wrong_order[:5].tolist())
    # got slot holding ref slot k's expert
    p = np.argmax(got_ids[:, None, :] == ref_ids[:, :, None], axis=2) if K > 0 else \
        np.zeros((T, 0), dtype=np.int64)
    return p


def check_routing(got_ids, got_gates, ref_ids, ref_gates, decided, gate_tol=1e-5):
    """Ids bit-exact up to the slot order of undecided tokens; gates within
    ``gate_tol`` after aligning slots.  Returns the slot permutation."""
    p = align_slots(got_ids, ref_ids, decided)
    g = np.take_along_axis(np.asarray(got_gates, dtype=np.float64), p, axis=1)
    assert np.max(np.abs(g - ref_gates), initial=0.0) < gate_tol
    return p


def aligned_slot_rows(got_slot_row, p):
    """The GPU's slot_row ([T*K]) with each token's slots put in the oracle's order."""
    T, K = p.shape
    return np.take_along_axis(np.asarray(got_slot_row).reshape(T, K), p, axis=1).reshape(-1)


TOKEN_TILE = 256   # token rows of one tile of the CTA-pair GEMMs


def tile_sample(offsets, perm_src, tile=TOKEN_TILE):
    """Tokens covering every `tile`-row token tile of every expert group: for
    each tile its first and last grouped row and the rows on either side of
    the middle of its MMA width (the boundary between the halves that the two
    CTAs of a pair load).  Returns sorted unique token indices."""
    rows = []
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        for t0 in range(lo, hi, tile):
            t1 = min(t0 + tile, hi)
            half = ((t1 - t0 + 15) & ~15) // 2
            for r in (t0, t1 - 1, t0 + half - 1, t0 + half):
                if t0 <= r < t1:
                    rows.append(r)
    return np.unique(np.asarray(perm_src)[np.asarray(rows, dtype=np.int64)])
