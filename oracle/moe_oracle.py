"""fp64 CPU oracle of the Mixtral sparse mixture-of-experts layer: the forward,
its backward with the routing held fixed, and the routing statistics.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import or run this module.
It shares no code with the CUDA library: it takes bf16 bit patterns
(``numpy.uint16``) straight from the input generator and widens them itself.

What it computes, step by step, and where each step is defined ("Mixtral of
Experts", arXiv 2401.04088):

* layer output: ``y = sum_i G(x)_i * E_i(x)`` over the n experts, and experts
  whose gate is zero need not be evaluated (§2.1, the layer-output sum and
  the sentence after it);
* gate: ``G(x) = Softmax(TopK(x . W_g))`` where ``TopK`` keeps the K largest of
  the n logits and sets the others to minus infinity (§2.1, the gating
  definition); Mixtral uses n = 8 and K = 2 (Table 1);
* expert: a SwiGLU feed-forward block (§2.1, the top-2 SwiGLU form of the
  layer).  The pages do not print the SwiGLU formula; the reading used here is
  ``E(x) = W2 (SiLU(W1 x) * (W3 x))`` with no biases, three dim x hidden
  matrices per expert, which is the reading that reproduces the 46.7B total /
  12.9B active parameter counts quoted for the model (the CPU tests check this
  against Table 1 and the quoted counts).

Readings where the pages are silent:

* ties in TopK go to the lower expert index; slot 0 holds the larger logit;
* the softmax runs over the K selected logits only (the others are minus
  infinity, so their exponentials are exactly zero);
* the routing structures are a stable counting sort of the flat assignments
  ``t*K + k`` by expert id (tokens ascending inside each expert group);
* the 32-layer stack applies ``x <- x + MoE(RMSNorm(x))`` with unit gain and
  eps = 1e-5, the normalised activations rounded to bf16 (not on the pages);
* the backward (the pages give no gradient) differentiates the layer output
  with the expert selection held fixed -- TopK is piecewise constant -- so the
  router weight and the input receive the gradient of the softmax over the
  selected logits (``moe_layer_backward``, pinned by central differences);
* the routing statistics (§5, Routing analysis: Fig. 7 and 9 expert shares,
  Table 5 repeated consecutive assignments) are returned as counts:
  per-(choice, expert) tokens, consecutive pairs with the same first choice
  and consecutive pairs whose K chosen experts intersect.

Precision: every input is widened exactly from bf16 to float64 and every step
runs in float64; nothing is rounded to a narrower type except where the method
itself defines a bf16 value (the RMSNorm output of the stack workload).  The
oracle has no mode that imitates the rounding points of any implementation.
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------- bf16 ----

def widen_bf16(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact: a bf16 is the top half of a float32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_bf16(values) -> np.ndarray:
    """float64 -> bf16 bit patterns, one round-to-nearest-even step.

    Finite values inside the bf16 normal range (or zero) only; the oracle never
    produces anything else.
    """
    v = np.ascontiguousarray(values, dtype=np.float64)
    bits = v.view(np.uint64)
    # Keep sign, 11 exponent bits and 7 mantissa bits of the float64; round the
    # 45 dropped mantissa bits to nearest, ties to even.  A mantissa carry
    # propagates into the exponent field, as rounding requires.
    lsb = (bits >> np.uint64(45)) & np.uint64(1)
    r = (bits + np.uint64((1 << 44) - 1) + lsb) >> np.uint64(45)
    sign = (r >> np.uint64(18)) & np.uint64(1)
    exp11 = (r >> np.uint64(7)) & np.uint64(0x7FF)
    mant = r & np.uint64(0x7F)
    zero = (bits & np.uint64(0x7FFFFFFFFFFFFFFF)) == 0
    exp8 = exp11.astype(np.int64) - 1023 + 127
    ok = zero | ((exp8 >= 1) & (exp8 <= 254))
    if not np.all(ok):
        raise ValueError("round_bf16: value outside the bf16 normal range")
    exp8 = np.where(zero, 0, exp8).astype(np.uint64)
    mant = np.where(zero, np.uint64(0), mant)
    out = (sign << np.uint64(15)) | (exp8 << np.uint64(7)) | mant
    return out.astype(np.uint16)


# ------------------------------------------------------------- router ----

def router_logits(x, w_gate) -> np.ndarray:
    """Logits l = x . W_g in float64 (§2.1, the gating definition).

    x: [T, dim] (bf16 bits or float64), w_gate: [dim, n]; returns [T, n].
    """
    return _f64(x) @ _f64(w_gate)


def topk_order(logits: np.ndarray) -> np.ndarray:
    """Expert indices of every token ordered by (logit descending, index ascending)."""
    # A stable sort of -l keeps equal logits in ascending index order.
    return np.argsort(-logits, axis=1, kind="stable")


def router(x, w_gate, top_k: int):
    """Top-K selection and gates (§2.1, the gating definition).

    Returns (ids [T, K] int64, gates [T, K] float64, logits [T, n]); slot k of
    a token holds its k-th largest logit, ties to the lower expert index, and
    the gates are the softmax of the K selected logits.
    """
    logits = router_logits(x, w_gate)
    ids = topk_order(logits)[:, :top_k]
    sel = np.take_along_axis(logits, ids, axis=1)
    return ids, softmax_selected(sel), logits


def softmax_selected(sel: np.ndarray) -> np.ndarray:
    """Softmax over the selected logits (the masked ones contribute exp(-inf) = 0)."""
    z = np.exp(sel - sel.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


# ------------------------------------------------------------- expert ----

def silu(a: np.ndarray) -> np.ndarray:
    """SiLU(a) = a * sigmoid(a) = a / (1 + exp(-a))."""
    return a / (1.0 + np.exp(-a))


def expert_weight_shapes(dim: int, hidden: int):
    """Shapes of the three matrices one SwiGLU expert reads: W1, W3, W2."""
    return [(hidden, dim), (hidden, dim), (dim, hidden)]


def expert_hidden(xr, w1, w3) -> np.ndarray:
    """SwiGLU activations SiLU(W1 x) * (W3 x) for the rows of ``xr`` ([m, dim] -> [m, hidden])."""
    xr, w1, w3 = _f64(xr), _f64(w1), _f64(w3)
    assert w1.shape == w3.shape and w1.shape[1] == xr.shape[1]
    return silu(xr @ w1.T) * (xr @ w3.T)


def expert_ffn(xr, w1, w3, w2) -> np.ndarray:
    """E(x) = W2 (SiLU(W1 x) * (W3 x)) applied to each row of ``xr`` ([m, dim] -> [m, dim])."""
    w2 = _f64(w2)
    s = expert_hidden(xr, w1, w3)
    assert w2.shape == (np.asarray(xr).shape[1], s.shape[1])
    return s @ w2.T


# ---------------------------------------------------------- the layer ----

def moe_layer(x, w_gate, w1, w3, w2, top_k: int):
    """Sparse MoE layer forward (§2.1, the top-2 SwiGLU form of the layer).

    x: [T, dim]; w_gate: [dim, n]; w1, w3: [n, hidden, dim]; w2: [n, dim, hidden].
    Each token evaluates only its K selected experts (experts with a zero gate
    are skipped).  Returns (y [T, dim] float64, ids [T, K], gates [T, K]).
    """
    xf = _f64(x)
    ids, gates, _ = router(xf, w_gate, top_k)
    T, dim = xf.shape
    n = np.asarray(w1).shape[0]
    y = np.zeros((T, dim))
    for e in range(n):                      # sum over the experts in index order
        tok, slot = np.nonzero(ids == e)
        if len(tok) == 0:
            continue
        out = expert_ffn(xf[tok], w1[e], w3[e], w2[e])
        y[tok] += gates[tok, slot][:, None] * out
    return y, ids, gates


def silu_grad(a: np.ndarray) -> np.ndarray:
    """d SiLU / da = sigmoid(a) * (1 + a * (1 - sigmoid(a)))."""
    sg = 1.0 / (1.0 + np.exp(-a))
    return sg * (1.0 + a * (1.0 - sg))


def moe_layer_backward(x, w_gate, w1, w3, w2, top_k: int, dy, weight_grads: bool = True):
    """Gradients of the sparse MoE layer (§2.1) for an upstream gradient dy.

    The routing (which K experts each token uses) is held fixed: TopK is
    piecewise constant, so the gradient reaches W_g and x only through the
    softmax of the selected logits.  With a = W1_e x, b = W3_e x, s = SiLU(a),
    h = s * b, o = W2_e h and y = sum_k g_k o_k:
      d o_k = g_k dy,          d g_k = <dy, o_k>,
      d h = W2_e^T d o,        d W2_e += d o h^T,
      d a = d h * b * SiLU'(a), d b = d h * s,
      d W1_e += d a x^T,       d W3_e += d b x^T,  d x += W1_e^T d a + W3_e^T d b,
      d l_k = g_k (d g_k - sum_j g_j d g_j)  (softmax over the selected logits),
      d W_g += x d l^T,        d x += W_g d l.
    Returns dict(dx [T, dim], dwg [dim, n], dw1, dw3 [n, hidden, dim],
    dw2 [n, dim, hidden]), float64.

    Every step is float64; nothing is rounded.
    weight_grads=False skips dw1 / dw3 / dw2 (returned as None), for callers
    that only need dx and dwg of a few tokens at full model size.
    """
    xf, wg = _f64(x), _f64(w_gate)
    g_up = _f64(dy)
    ids, gates, _ = router(xf, wg, top_k)
    T, dim = xf.shape
    n = np.asarray(w1).shape[0]
    dx = np.zeros_like(xf)
    dwg = np.zeros_like(wg)
    dw1 = dw3 = dw2 = None
    if weight_grads:
        dw1 = np.zeros(np.asarray(w1).shape)
        dw3 = np.zeros(np.asarray(w3).shape)
        dw2 = np.zeros(np.asarray(w2).shape)
    dgate = np.zeros((T, top_k))
    for e in range(n):
        tok, slot = np.nonzero(ids == e)
        if len(tok) == 0:
            continue
        W1e, W3e, W2e = _f64(w1[e]), _f64(w3[e]), _f64(w2[e])   # one expert at a time
        xe = xf[tok]
        a = xe @ W1e.T
        b = xe @ W3e.T
        s = silu(a)
        h = s * b
        o = h @ W2e.T
        do = gates[tok, slot][:, None] * g_up[tok]
        dgate[tok, slot] = np.sum(g_up[tok] * o, axis=1)
        dh = do @ W2e
        da = dh * b * silu_grad(a)
        db = dh * s
        if weight_grads:
            dw2[e] += do.T @ h
            dw1[e] += da.T @ xe
            dw3[e] += db.T @ xe
        np.add.at(dx, tok, da @ W1e + db @ W3e)
    dl_sel = gates * (dgate - np.sum(gates * dgate, axis=1, keepdims=True))
    dl = np.zeros((T, n))
    np.put_along_axis(dl, ids, dl_sel, axis=1)
    dwg += xf.T @ dl
    dx += dl @ wg.T
    return dict(dx=dx, dwg=dwg, dw1=dw1, dw3=dw3, dw2=dw2)


def expert_weight_grad_units(x, w_gate, w1, w3, w2, top_k: int, dy, e: int, units):
    """Expert e's weight gradients for a few hidden units j in ``units``, from the
    same chain rule as ``moe_layer_backward`` (routing fixed, exact mode) but
    evaluated on hidden units j only: dW1_e[j, :] and dW3_e[j, :] (rows of the
    [hidden, dim] gradients) and dW2_e[:, j] (columns of the [dim, hidden]
    gradient).  Hidden unit j of the expert needs only a_j = W1_e[j] x,
    b_j = W3_e[j] x and dh_j = W2_e[:, j] . d o for the tokens routed to e,
    so the cost is a few dot products per token and unit, at any model size.
    Returns dict(dw1 [len(units), dim], dw3 [len(units), dim],
    dw2 [dim, len(units)]), float64.
    """
    units = np.asarray(units)
    xf, wg = _f64(x), _f64(w_gate)
    g_up = _f64(dy)
    ids, gates, _ = router(xf, wg, top_k)
    tok, slot = np.nonzero(ids == e)
    W1j = _f64(np.asarray(w1)[e][units])            # [u, dim]
    W3j = _f64(np.asarray(w3)[e][units])            # [u, dim]
    W2j = _f64(np.asarray(w2)[e][:, units])         # [dim, u]
    xe = xf[tok]
    a = xe @ W1j.T
    b = xe @ W3j.T
    h = silu(a) * b
    do = gates[tok, slot][:, None] * g_up[tok]
    dh = do @ W2j
    da = dh * b * silu_grad(a)
    db = dh * silu(a)
    return dict(dw1=da.T @ xe, dw3=db.T @ xe, dw2=do.T @ h)


def rmsnorm_bf16(x, eps: float) -> np.ndarray:
    """bf16 bits of x / sqrt(mean(x^2) + eps) per row (unit gain; stack workload only)."""
    xf = _f64(x)
    r = np.sqrt((xf * xf).mean(axis=1, keepdims=True) + eps)
    return round_bf16(xf / r)


def stack_layer(x_bits, w_gate, w1, w3, w2, top_k: int, eps: float):
    """One residual block of the stack: x + MoE(RMSNorm(x)), float64 (not bf16-rounded)."""
    u = rmsnorm_bf16(x_bits, eps)
    y, ids, gates = moe_layer(u, w_gate, w1, w3, w2, top_k)
    return _f64(x_bits) + y, ids, gates, u


# ---------------------------------------------- the layer, step by step ----

def routing_tables(ids: np.ndarray, n_experts: int):
    """Expert-grouped permutation of the flat assignments a = t*K + k.

    counts[e]   number of assignments to expert e;
    offsets     exclusive prefix sum of counts, length n + 1;
    perm_src[r] token of the assignment stored at grouped row r (stable: tokens
                ascending inside each expert group);
    slot_row[a] grouped row of assignment a (the inverse permutation).
    """
    flat = np.asarray(ids).reshape(-1)
    K = np.asarray(ids).shape[1]
    counts = np.bincount(flat, minlength=n_experts).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    order = np.argsort(flat, kind="stable")      # grouped row -> flat assignment
    perm_src = order // K
    slot_row = np.empty_like(order)
    slot_row[order] = np.arange(len(order))
    return counts, offsets, perm_src, slot_row


def routing_stats(ids: np.ndarray, n_experts: int):
    """Routing statistics of "Mixtral of Experts" section 5 (Routing analysis).

    slot_counts[k, e]  tokens whose k-th choice is expert e (Fig. 7 counts the
                       first or second choice, i.e. the sum over k; Fig. 9
                       splits it by choice);
    first_repeat       pairs of consecutive tokens (t, t+1) with the same first
                       choice (Table 5, "first choice only");
    any_repeat         pairs whose sets of K chosen experts share at least one
                       expert (Table 5, "first or second choice" for K = 2);
    pairs              T - 1 consecutive pairs (0 when T < 2).
    """
    ids = np.asarray(ids)
    T, K = ids.shape
    slot_counts = np.zeros((K, n_experts), dtype=np.int64)
    for k in range(K):
        for t in range(T):
            slot_counts[k, ids[t, k]] += 1
    first_repeat = 0
    any_repeat = 0
    for t in range(T - 1):
        if ids[t, 0] == ids[t + 1, 0]:
            first_repeat += 1
        if set(ids[t].tolist()) & set(ids[t + 1].tolist()):
            any_repeat += 1
    return dict(slot_counts=slot_counts, first_repeat=first_repeat, any_repeat=any_repeat,
                pairs=max(T - 1, 0))


def grouped_ffn(x_perm, offsets, w1, w3, w2):
    """Expert FFN over grouped rows: rows [offsets[e], offsets[e+1]) use expert e.

    Returns (y_perm [R, dim], hidden activations [R, hidden]), float64.
    """
    xp = _f64(x_perm)
    n = len(offsets) - 1
    hidden = np.asarray(w1).shape[1]
    y_perm = np.zeros_like(xp)
    hid = np.zeros((xp.shape[0], hidden))
    for e in range(n):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            hid[lo:hi] = expert_hidden(xp[lo:hi], w1[e], w3[e])
            y_perm[lo:hi] = hid[lo:hi] @ _f64(w2[e]).T
    return y_perm, hid


def combine(y_perm, slot_row, gates, residual=None) -> np.ndarray:
    """y[t] = sum_k gates[t, k] * y_perm[slot_row[t*K + k]] (+ residual[t]), float64."""
    yp = _f64(y_perm)
    g = np.asarray(gates, dtype=np.float64)
    T, K = g.shape
    rows = np.asarray(slot_row).reshape(T, K)
    y = np.zeros((T, yp.shape[1]))
    for k in range(K):
        y += g[:, k:k + 1] * yp[rows[:, k]]
    if residual is not None:
        y += _f64(residual)
    return y


def _f64(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return widen_bf16(a)
    return a.astype(np.float64, copy=False)
