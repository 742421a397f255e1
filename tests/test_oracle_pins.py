"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test names what it pins: values printed on the pages (golden fixtures,
cited inside them), closed forms, special cases that reduce to textbook
values, invariants of the definition, and brute force on tiny inputs.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import moe_inputs as mi
from oracle import moe_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand_layer(rng, T, d, h, n, scale_x=1.0):
    """Small float64 layer (values exactly representable as bf16)."""
    def bf(a):
        return orc.widen_bf16(orc.round_bf16(a))
    x = bf(rng.standard_normal((T, d)) * scale_x)
    wg = bf(rng.standard_normal((d, n)) / np.sqrt(d))
    w1 = bf(rng.standard_normal((n, h, d)) / np.sqrt(d))
    w3 = bf(rng.standard_normal((n, h, d)) / np.sqrt(d))
    w2 = bf(rng.standard_normal((n, d, h)) / np.sqrt(h))
    return x, wg, w1, w3, w2


# ------------------------------------------------------------ bf16 -------

def test_widen_bf16_bit_patterns():
    # IEEE bfloat16: sign 1, exponent 8 (bias 127), mantissa 7.
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0001, 0x7F7F, 0x0000, 0x8000, 0x4049],
                    dtype=np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 2.0 ** -133, (2 - 2.0 ** -7) * 2.0 ** 127,
            0.0, -0.0, 3.140625]
    got = orc.widen_bf16(bits)
    assert list(got) == want


def test_round_bf16_nearest_even():
    vals = np.array([1.0, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -30,
                     -2.0, 3.14159265358979, 0.0, 1e-30])
    want = [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xC000, 0x4049, 0x0000, 0x0DA2]
    assert [int(v) for v in orc.round_bf16(vals)] == want
    # agrees with an independent float32 -> bf16 rounding on float32-exact values
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(100000) * 10.0 ** rng.integers(-5, 5, 100000)).astype(np.float32)
    assert np.array_equal(orc.round_bf16(v.astype(np.float64)), mi.f32_to_bf16(v))


# ---------------------------------------------------------- router -------

def test_router_orientation_hand_example():
    # W_g [dim=4, n=3] picks coordinates: l = (x0, x1, x2); x3 is ignored.
    wg = np.zeros((4, 3))
    wg[0, 0] = wg[1, 1] = wg[2, 2] = 1.0
    x = np.array([[0.5, 2.0, -1.0, 7.0]])
    ids, gates, logits = orc.router(x, wg, 2)
    assert logits.tolist() == [[0.5, 2.0, -1.0]]
    assert ids.tolist() == [[1, 0]]
    g0 = 1.0 / (1.0 + math.exp(-1.5))          # e^2 / (e^2 + e^0.5)
    assert abs(gates[0, 0] - g0) < 1e-15 and abs(gates[0, 1] - (1 - g0)) < 1e-15


def test_topk_brute_force_all_subsets():
    rng = np.random.default_rng(1)
    for n, K in [(8, 2), (8, 1), (5, 3), (8, 8), (1, 1)]:
        logits = rng.integers(-3, 4, size=(300, n)).astype(np.float64)  # many exact ties
        ids = orc.topk_order(logits)[:, :K]
        for t in range(logits.shape[0]):
            best = None
            for sub in itertools.combinations(range(n), K):
                key = (-sum(logits[t, list(sub)]), sub)   # max sum, then lowest indices
                if best is None or key < best:
                    best = key
            assert sorted(ids[t].tolist()) == list(best[1])
            # slot order: logits non-increasing, equal logits by ascending index
            sl = logits[t, ids[t]]
            for k in range(K - 1):
                assert sl[k] > sl[k + 1] or (sl[k] == sl[k + 1] and ids[t, k] < ids[t, k + 1])


def test_topk_many_experts_by_pairwise_counting():
    """Fine-grained routing (top 8 of 160, the pages' example): expert e is in
    slot k exactly when k experts beat it, where j beats e if its logit is
    larger or equal with a lower index (an O(n^2) restatement of the order,
    independent of the oracle's sort)."""
    rng = np.random.default_rng(4)
    for n, K in [(160, 8), (64, 6), (256, 8), (40, 1)]:
        logits = rng.integers(-6, 7, size=(60, n)).astype(np.float64)  # many exact ties
        ids = orc.topk_order(logits)[:, :K]
        for t in range(logits.shape[0]):
            l = logits[t]
            beaten_by = ((l[None, :] > l[:, None]) |
                         ((l[None, :] == l[:, None]) & (np.arange(n)[None, :] < np.arange(n)[:, None])))
            rank = beaten_by.sum(1)            # experts that beat e
            expect = np.argsort(rank)[:K]      # ranks are a permutation of 0..n-1
            assert np.array_equal(ids[t], expect)
            assert np.array_equal(rank[ids[t]], np.arange(K))


def test_forced_tie_goes_to_lower_index():
    x = np.zeros((3, 16))
    wg = np.random.default_rng(2).standard_normal((16, 8))
    ids, gates, _ = orc.router(x, wg, 2)
    assert ids.tolist() == [[0, 1]] * 3
    assert np.all(gates == 0.5)


def test_gates_invariants_and_k2_closed_form():
    rng = np.random.default_rng(3)
    x, wg, *_ = _rand_layer(rng, 500, 64, 8, 8)
    for K in (1, 2, 3, 8):
        ids, gates, logits = orc.router(x, wg, K)
        assert np.all(gates >= 0)
        assert np.allclose(gates.sum(1), 1.0, atol=1e-12, rtol=0)
    ids, gates, logits = orc.router(x, wg, 2)
    l0 = np.take_along_axis(logits, ids[:, :1], 1)[:, 0]
    l1 = np.take_along_axis(logits, ids[:, 1:2], 1)[:, 0]
    # two-way softmax: g0 = 1 / (1 + exp(l1 - l0)), the logistic function of the gap
    assert np.allclose(gates[:, 0], 1.0 / (1.0 + np.exp(l1 - l0)), atol=1e-15, rtol=0)
    assert np.all(gates[:, 0] >= 0.5)


# ---------------------------------------------------------- expert -------

def test_silu_textbook_values():
    e = math.e
    got = orc.silu(np.array([0.0, 1.0, -1.0, 2.0, 40.0, -40.0]))
    want = [0.0, e / (1 + e), -1 / (1 + e), 2 * e * e / (1 + e * e), 40.0, 0.0]
    assert np.allclose(got, want, atol=1e-15, rtol=1e-15)


def test_swiglu_hand_example_orientation():
    # dim = hidden = 2, permutation-like matrices so every operand orientation matters:
    # W1 x = (x1, 0), W3 x = (x0, x1), W2 s = (3 s1, 2 s0)
    w1 = np.array([[0.0, 1.0], [0.0, 0.0]])
    w3 = np.array([[1.0, 0.0], [0.0, 1.0]])
    w2 = np.array([[0.0, 3.0], [2.0, 0.0]])
    x = np.array([[5.0, 1.0]])
    s0 = (1.0 * math.e / (1 + math.e)) * 5.0      # SiLU(x1) * x0 with x1 = 1
    want = np.array([[0.0, 2.0 * s0]])
    got = orc.expert_ffn(x, w1, w3, w2)
    assert np.allclose(got, want, atol=1e-14, rtol=0)
    # non-square: dim 2, hidden 3
    w1 = np.array([[1.0, 0.0], [0.0, 0.0], [0.0, -1.0]])
    w3 = np.array([[0.0, 1.0], [1.0, 1.0], [1.0, 0.0]])
    w2 = np.array([[1.0, 0.0, 0.0], [0.0, 0.0, 1.0]])
    x = np.array([[2.0, 3.0]])
    # a = (2, 0, -3), b = (3, 5, 2); s = (SiLU(2)*3, 0, SiLU(-3)*2); y = (s0, s2)
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))
    want = np.array([[2 * sig(2) * 3, -3 * sig(-3) * 2]])
    assert np.allclose(orc.expert_ffn(x, w1, w3, w2), want, atol=1e-14, rtol=0)


def test_expert_has_three_dim_by_hidden_matrices_param_count():
    """Table 1 plus a three-matrix SwiGLU expert reproduces the quoted 46.7B / 47B / 13B."""
    t = _golden("mixtral_table1.json")
    d, h, n, K = t["dim"], t["hidden_dim"], t["num_experts"], t["top_k_experts"]
    expert = sum(a * b for a, b in orc.expert_weight_shapes(d, h))
    attn = d * (t["n_heads"] * t["head_dim"]) * 2 + d * (t["n_kv_heads"] * t["head_dim"]) * 2
    router = d * n
    norms = 2 * d
    per_layer_total = attn + router + norms + n * expert
    per_layer_active = attn + router + norms + K * expert
    emb = 2 * t["vocab_size"] * d + d          # input embedding, output head, final norm
    total = t["n_layers"] * per_layer_total + emb
    active = t["n_layers"] * per_layer_active + emb
    assert round(total / 1e9) == t["total_params_billion_rounded"]
    assert round(total / 1e8) / 10 == t["total_params_billion_one_decimal"]
    assert round(active / 1e9) == t["active_params_billion_rounded"]
    # the expert really consumes exactly those shapes
    rng = np.random.default_rng(4)
    dd, hh = 6, 10
    shapes = orc.expert_weight_shapes(dd, hh)
    ws = [rng.standard_normal(s) for s in shapes]
    assert orc.expert_ffn(rng.standard_normal((3, dd)), *ws).shape == (3, dd)


# ----------------------------------------------------------- layer -------

def _dense_masked_reference(x, wg, w1, w3, w2, K):
    """The layer as printed: every expert evaluated, gate = softmax of the -inf-masked logits."""
    logits = x @ wg
    n = wg.shape[1]
    out = np.zeros_like(x)
    for t in range(x.shape[0]):
        l = logits[t]
        kth = sorted(range(n), key=lambda i: (-l[i], i))[:K]
        masked = np.full(n, -np.inf)
        masked[kth] = l[kth]
        g = np.exp(masked - masked.max())
        g = g / g.sum()
        for i in range(n):
            a = w1[i] @ x[t]
            b = w3[i] @ x[t]
            s = a / (1 + np.exp(-a)) * b
            out[t] += g[i] * (w2[i] @ s)
    return out


@pytest.mark.parametrize("n,K", [(8, 2), (8, 1), (4, 3), (8, 8), (1, 1), (160, 8)])
def test_sparse_equals_dense_masked_sum(n, K):
    rng = np.random.default_rng(10 + n * 10 + K)
    x, wg, w1, w3, w2 = _rand_layer(rng, 24, 16, 12, n)
    y, ids, gates = orc.moe_layer(x, wg, w1, w3, w2, K)
    ref = _dense_masked_reference(x, wg, w1, w3, w2, K)
    assert np.max(np.abs(y - ref)) < 1e-12


@pytest.mark.parametrize("K", [1, 2, 8])
def test_identical_experts_reduce_to_dense_ffn(K):
    """Upcycled experts (all copies of one FFN): gates sum to 1, so y = FFN(x)."""
    rng = np.random.default_rng(20 + K)
    x, wg, w1, w3, w2 = _rand_layer(rng, 16, 16, 24, 1)
    n = 8
    W1, W3, W2 = (np.repeat(w, n, 0) for w in (w1, w3, w2))
    wg = rng.standard_normal((16, n))
    y, _, _ = orc.moe_layer(x, wg, W1, W3, W2, K)
    ffn = orc.expert_ffn(x, w1[0], w3[0], w2[0])
    assert np.max(np.abs(y - ffn)) < 1e-12


def test_single_expert_is_swiglu():
    rng = np.random.default_rng(30)
    x, wg, w1, w3, w2 = _rand_layer(rng, 10, 8, 12, 1)
    y, ids, gates = orc.moe_layer(x, wg, w1, w3, w2, 1)
    assert np.all(ids == 0) and np.all(gates == 1.0)
    a = x @ w1[0].T
    b = x @ w3[0].T
    want = (a * (1.0 / (1.0 + np.exp(-a))) * b) @ w2[0].T
    assert np.max(np.abs(y - want)) < 1e-13


def test_stepwise_path_equals_layer():
    """router -> grouping -> grouped FFN -> combine composes to the layer."""
    rng = np.random.default_rng(40)
    x, wg, w1, w3, w2 = _rand_layer(rng, 50, 16, 12, 8)
    y, ids, gates = orc.moe_layer(x, wg, w1, w3, w2, 2)
    counts, offsets, perm_src, slot_row = orc.routing_tables(ids, 8)
    y_perm, _ = orc.grouped_ffn(x[perm_src], offsets, w1, w3, w2)
    y2 = orc.combine(y_perm, slot_row, gates)
    assert np.max(np.abs(y - y2)) < 1e-12


# --------------------------------------------------------- grouping -------

def test_routing_tables_brute_force():
    rng = np.random.default_rng(50)
    for T, n, K in [(1, 8, 2), (37, 8, 2), (64, 5, 3), (20, 1, 1), (9, 8, 8)]:
        ids = np.stack([rng.permutation(n)[:K] for _ in range(T)])
        counts, offsets, perm_src, slot_row = orc.routing_tables(ids, n)
        assert counts.sum() == T * K and offsets[0] == 0 and offsets[-1] == T * K
        assert np.all(np.diff(offsets) >= 0)
        rows = []
        for e in range(n):                       # brute force: tokens ascending per expert
            for t in range(T):
                for k in range(K):
                    if ids[t, k] == e:
                        rows.append((t, k))
        assert len(rows) == T * K
        for r, (t, k) in enumerate(rows):
            assert perm_src[r] == t
            assert slot_row[t * K + k] == r
        assert sorted(slot_row.tolist()) == list(range(T * K))


def test_rmsnorm_closed_form():
    x = orc.round_bf16(np.array([[3.0, 4.0], [2.0, 2.0]]))
    u = orc.widen_bf16(orc.rmsnorm_bf16(x, 0.0))
    r = math.sqrt(12.5)
    want = orc.widen_bf16(orc.round_bf16(np.array([[3 / r, 4 / r], [1.0, 1.0]])))
    assert np.array_equal(u, want)


# ------------------------------------------------------ statistics -------

def test_random_routing_matches_printed_expectations():
    """iid tokens and a random router: shares ~ 1/8 (Fig. 7) and the Table 5 random
    repeat rates (12.5% first choice, 1-(6/8)(5/7) ~ 46% either choice)."""
    g = _golden("routing_random_expectations.json")
    cfg = mi.Config("stats", T=20000, dim=1024, hidden=128, seed=4242)
    x = mi.gen_x(cfg)
    wg = mi.gen_router_weight(cfg)
    ids, _, _ = orc.router(x, wg, g["top_k"])
    share = np.bincount(ids.reshape(-1), minlength=8) / ids.size
    assert np.all(np.abs(share - g["uniform_share"]) < 0.02)
    first = np.mean(ids[1:, 0] == ids[:-1, 0])
    either = np.mean([len(set(a) & set(b)) > 0 for a, b in zip(ids[1:], ids[:-1])])
    exp_either = 1 - (6 / 8) * (5 / 7)
    assert round(exp_either * 100) == g["first_or_second_repeat_printed_percent"]
    assert abs(first - g["first_choice_repeat"]) < 0.015
    assert abs(either - exp_either) < 0.025


def test_routing_stats_hand_example_and_random_expectations():
    """Table 5 statistics: a hand-worked sequence, then iid tokens against the
    printed random expectations (12.5 % first choice, 1-(6/8)(5/7) ~ 46 %)."""
    ids = np.array([[0, 1], [0, 2], [3, 1], [4, 5], [5, 4], [5, 6]])
    st = orc.routing_stats(ids, 8)
    # pairs (0,1): same first choice; (1,2): no shared expert; (2,3): none;
    # (3,4): share 4 and 5; (4,5): same first choice 5
    assert st["pairs"] == 5
    assert st["first_repeat"] == 2
    assert st["any_repeat"] == 3
    assert st["slot_counts"][0].tolist() == [2, 0, 0, 1, 1, 2, 0, 0]
    assert st["slot_counts"][1].tolist() == [0, 2, 1, 0, 1, 1, 1, 0]
    g = _golden("routing_random_expectations.json")
    rng = np.random.default_rng(5)
    ids = np.stack([rng.permutation(8)[:2] for _ in range(20000)])
    st = orc.routing_stats(ids, 8)
    assert abs(st["first_repeat"] / st["pairs"] - g["first_choice_repeat"]) < 0.01
    assert abs(st["any_repeat"] / st["pairs"] - (1 - (6 / 8) * (5 / 7))) < 0.015
    share = st["slot_counts"].sum(0) / ids.size
    assert np.all(np.abs(share - g["uniform_share"]) < 0.01)


def test_stack_layer_residual_and_zero_experts():
    """x + MoE(RMSNorm(x)): with W2 = 0 every expert outputs 0, so the block is the
    identity; with identical experts it is x + FFN(RMSNorm(x))."""
    rng = np.random.default_rng(60)
    x, wg, w1, w3, w2 = _rand_layer(rng, 12, 16, 8, 4)
    xb = orc.round_bf16(x)
    out, _, _, _ = orc.stack_layer(xb, wg, w1, w3, np.zeros_like(w2), 2, 1e-5)
    assert np.array_equal(out, orc.widen_bf16(xb))
    W1, W3, W2 = (np.repeat(w[:1], 4, 0) for w in (w1, w3, w2))
    out, _, _, u = orc.stack_layer(xb, wg, W1, W3, W2, 2, 1e-5)
    want = orc.widen_bf16(xb) + orc.expert_ffn(orc.widen_bf16(u), w1[0], w3[0], w2[0])
    assert np.max(np.abs(out - want)) < 1e-12


# ---------------------------------------------------------- backward -----

def _loss(x, wg, w1, w3, w2, K, dy):
    y, _, _ = orc.moe_layer(x, wg, w1, w3, w2, K)
    return float(np.sum(y * dy))


@pytest.mark.parametrize("n,K", [(8, 2), (4, 1), (5, 3)])
def test_backward_matches_central_differences(n, K):
    """Every gradient of the oracle's backward against central finite differences
    of the forward (routing fixed: inputs whose top-K margin exceeds the step)."""
    rng = np.random.default_rng(60 + n + K)
    T, d, h = 5, 6, 7
    x, wg, w1, w3, w2 = (rng.standard_normal(s) for s in
                         [(T, d), (d, n), (n, h, d), (n, h, d), (n, d, h)])
    dy = rng.standard_normal((T, d))
    srt = -np.sort(-orc.router_logits(x, wg), axis=1)
    if K < n:
        assert np.min(srt[:, K - 1] - srt[:, K]) > 1e-3   # routing stays fixed under the step
    g = orc.moe_layer_backward(x, wg, w1, w3, w2, K, dy)
    eps = 1e-6
    for name, arr in [("dx", x), ("dwg", wg), ("dw1", w1), ("dw3", w3), ("dw2", w2)]:
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = _loss(x, wg, w1, w3, w2, K, dy)
            arr[idx] = old - eps
            lm = _loss(x, wg, w1, w3, w2, K, dy)
            arr[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        assert np.max(np.abs(num - g[name])) < 1e-6 * (1 + np.max(np.abs(num))), name


def test_backward_single_expert_is_the_dense_swiglu_gradient():
    """n = 1, K = 1: the gate is 1 and constant, so dW_g = 0 and every other
    gradient is the plain SwiGLU FFN's (written here with the chain rule on
    explicit per-element loops)."""
    rng = np.random.default_rng(70)
    T, d, h = 3, 4, 5
    x = rng.standard_normal((T, d))
    wg = rng.standard_normal((d, 1))
    w1, w3 = rng.standard_normal((1, h, d)), rng.standard_normal((1, h, d))
    w2 = rng.standard_normal((1, d, h))
    dy = rng.standard_normal((T, d))
    g = orc.moe_layer_backward(x, wg, w1, w3, w2, 1, dy)
    assert np.all(g["dwg"] == 0)
    dx = np.zeros((T, d))
    dw2 = np.zeros((d, h))
    for t in range(T):
        a = [sum(w1[0, j, i] * x[t, i] for i in range(d)) for j in range(h)]
        b = [sum(w3[0, j, i] * x[t, i] for i in range(d)) for j in range(h)]
        sig = [1 / (1 + math.exp(-v)) for v in a]
        hh = [a[j] * sig[j] * b[j] for j in range(h)]
        dh = [sum(dy[t, i] * w2[0, i, j] for i in range(d)) for j in range(h)]
        for i in range(d):
            for j in range(h):
                dw2[i, j] += dy[t, i] * hh[j]
        for j in range(h):
            da = dh[j] * b[j] * sig[j] * (1 + a[j] * (1 - sig[j]))
            db = dh[j] * a[j] * sig[j]
            for i in range(d):
                dx[t, i] += da * w1[0, j, i] + db * w3[0, j, i]
    assert np.max(np.abs(dx - g["dx"])) < 1e-12
    assert np.max(np.abs(dw2 - g["dw2"][0])) < 1e-12


def test_gpu_rounding_model_stays_near_exact():
    """The model of the CUDA backward's bf16 storage points (test code, not the
    oracle) differs from the exact oracle by bf16-sized amounts only."""
    from tests.gpu_rounding_model import backward_at_gpu_storage_points
    rng = np.random.default_rng(71)
    x, wg, w1, w3, w2 = _rand_layer(rng, 40, 16, 24, 8)
    dy = orc.widen_bf16(orc.round_bf16(rng.standard_normal((40, 16))))
    a = orc.moe_layer_backward(x, wg, w1, w3, w2, 2, dy)
    b = backward_at_gpu_storage_points(x, wg, w1, w3, w2, 2, dy)
    for k in a:
        rms = np.sqrt(np.mean(a[k] ** 2))
        assert np.max(np.abs(a[k] - b[k])) < 0.1 * rms, k
        assert np.max(np.abs(a[k] - b[k])) > 0, k


def test_gpu_rounding_model_is_exact_where_nothing_rounds():
    """With every intermediate exactly representable in bf16 (small integers
    and zero router weight), the storage-point model equals the exact oracle."""
    from tests.gpu_rounding_model import backward_at_gpu_storage_points
    T, d, h = 3, 2, 2
    x = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    wg = np.zeros((d, 1))
    w1 = np.full((1, h, d), 0.0)          # a = 0: SiLU(0) = 0, SiLU'(0) = 1/2
    w3 = np.array([[[1.0, 0.0], [0.0, 2.0]]])
    w2 = np.array([[[1.0, 1.0], [0.0, 1.0]]])
    dy = np.array([[1.0, 2.0], [0.5, 0.0], [1.0, 1.0]])
    a = orc.moe_layer_backward(x, wg, w1, w3, w2, 1, dy)
    b = backward_at_gpu_storage_points(x, wg, w1, w3, w2, 1, dy)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_backward_unit_gradients_match_the_full_backward():
    # the per-unit weight gradients (used to check large batches on sampled
    # units) against the full backward, itself pinned by central differences
    cfg = mi.Config("units", T=40, dim=16, hidden=24, n_experts=6, top_k=2, seed=4711)
    L = mi.make_layer(cfg)
    dy = mi.gen_x(cfg.replace(seed=4712))
    full = orc.moe_layer_backward(L.x, L.wg, L.w1, L.w3, L.w2, 2, dy)
    ids, _, _ = orc.router(L.x, L.wg, 2)
    for e in range(cfg.n_experts):
        units = [0, 5, 23] if e % 2 == 0 else [7, 11]
        got = orc.expert_weight_grad_units(L.x, L.wg, L.w1, L.w3, L.w2, 2, dy, e, units)
        scale = max(np.abs(full["dw1"]).max(), 1e-30)
        assert np.allclose(got["dw1"], full["dw1"][e][units], rtol=1e-12, atol=1e-14 * scale)
        assert np.allclose(got["dw3"], full["dw3"][e][units], rtol=1e-12, atol=1e-14 * scale)
        assert np.allclose(got["dw2"], full["dw2"][e][:, units], rtol=1e-12, atol=1e-14 * scale)
        if not np.any(ids == e):              # an expert with no tokens: zero gradients
            assert not np.any(got["dw1"]) and not np.any(got["dw2"])
    part = orc.moe_layer_backward(L.x, L.wg, L.w1, L.w3, L.w2, 2, dy, weight_grads=False)
    assert part["dw1"] is None and part["dw2"] is None
    assert np.array_equal(part["dx"], full["dx"]) and np.array_equal(part["dwg"], full["dwg"])
