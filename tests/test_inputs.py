"""The shared input generator: determinism, C/numpy agreement, distributions."""
import numpy as np

import moe_inputs as mi
from tests.inputs_filtered import (TOKEN_TILE, align_slots, ambiguous_tokens, filtered_layer,
                                   tile_sample)


def test_c_and_numpy_streams_agree():
    tab = mi.normal_table(1.0)
    key = mi.stream_key(46001, mi.T_X, 3, 1)
    for start in (0, 12345, (1 << 32) - 100):
        a = mi.fill(5000, start, key, tab, use_c=True)
        b = mi.fill(5000, start, key, tab, use_c=False)
        assert np.array_equal(a, b)
    rows = np.array([5, 0, 77])
    r = mi.fill_rows(rows, 64, key, tab)
    full = mi.fill(78 * 64, 0, key, tab).reshape(78, 64)
    assert np.array_equal(r, full[rows])


def test_streams_are_distinct_and_deterministic():
    tab = mi.normal_table(1.0)
    a = mi.fill(1000, 0, mi.stream_key(1, 3, 0, 0), tab)
    b = mi.fill(1000, 0, mi.stream_key(1, 3, 0, 1), tab)
    c = mi.fill(1000, 0, mi.stream_key(1, 3, 0, 0), tab)
    assert np.array_equal(a, c) and not np.array_equal(a, b)


def test_normal_table_moments():
    for scale in (1.0, 1 / 64.0, 1 / np.sqrt(14336)):
        v = mi.bf16_to_f32(mi.normal_table(scale)).astype(np.float64)
        assert abs(v.mean()) < 1e-3 * scale
        assert abs(v.std() / scale - 1.0) < 5e-3
        assert np.all(np.diff(v) >= 0)


def test_tiny_layer_shapes_and_scales():
    L = mi.make_layer(mi.CONFIGS["tiny"])
    cfg = L.cfg
    assert L.x.shape == (64, 128) and L.wg.shape == (128, 8)
    assert L.w1.shape == (8, 256, 128) and L.w2.shape == (8, 128, 256)
    assert abs(mi.bf16_to_f32(L.w1).std() * np.sqrt(cfg.dim) - 1) < 0.02
    assert abs(mi.bf16_to_f32(L.w2).std() * np.sqrt(cfg.hidden) - 1) < 0.02


def test_gap_filter_removes_ambiguous_tokens():
    cfg = mi.CONFIGS["tiny"].replace(T=4000)
    L = filtered_layer(cfg, experts=False)
    assert L.redrawn > 0
    assert not ambiguous_tokens(L.x, L.wg, cfg.top_k).any()


def test_zipf_calibration():
    p = mi.zipf_shares(8, 1.2)
    assert abs(p[0] - 0.4286) < 1e-3
    b = mi.calibrate_bias(p)
    assert np.max(np.abs(mi.gaussian_argmax_probs(b) - p)) < 5e-4


def test_skewed_tokens_follow_zipf_top1():
    from oracle import moe_oracle as orc
    cfg = mi.CONFIGS["skew"].replace(T=8192, dim=512, hidden=128)
    L = mi.make_layer(cfg, experts=False)
    ids, _, _ = orc.router(L.x, L.wg, 2)
    share = np.bincount(ids[:, 0], minlength=8) / cfg.T
    assert np.max(np.abs(share - mi.zipf_shares(8, 1.2))) < 0.03
    assert 0.38 < share[0] < 0.48


def test_tile_sample_covers_every_tile():
    # the full-size parity sampler on a hand-built grouping: experts of 0, 1,
    # 256, 257 and 600 rows; every tile must contribute its first and last row
    counts = np.array([0, 1, 256, 257, 600])
    offsets = np.concatenate([[0], np.cumsum(counts)])
    perm_src = np.arange(offsets[-1])          # identity: token == grouped row
    toks = set(tile_sample(offsets, perm_src).tolist())
    n_tiles = 0
    for e in range(len(counts)):
        for t0 in range(offsets[e], offsets[e + 1], TOKEN_TILE):
            t1 = min(t0 + TOKEN_TILE, offsets[e + 1])
            assert t0 in toks and t1 - 1 in toks
            n_tiles += 1
    assert n_tiles == 0 + 1 + 1 + 2 + 3
    assert offsets[-1] - 1 in toks             # the last row of the last partial tile
    assert 1 + 256 + 128 in toks               # both sides of the middle of a full tile


def test_align_slots_accepts_only_reordered_undecided_tokens():
    import pytest
    ref = np.array([[0, 1], [2, 3], [4, 5]])
    got = np.array([[0, 1], [3, 2], [4, 5]])
    p = align_slots(got, ref, np.array([True, False, True]))
    assert p.tolist() == [[0, 1], [1, 0], [0, 1]]
    with pytest.raises(AssertionError):        # order decided: a swap is an error
        align_slots(got, ref, np.array([True, True, True]))
    with pytest.raises(AssertionError):        # another expert is always an error
        align_slots(np.array([[0, 1], [2, 6], [4, 5]]), ref, np.array([False] * 3))
