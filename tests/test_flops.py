"""FLOP accounting of the throughput metric (host arithmetic, no GPU):
executed FLOPs credit the query-major cover at 4 d (forward) and 10 d
(backward) per covered entry, issued FLOPs count the GEMMs the kernels run,
dense FLOPs count the causal mask."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from dynamic_vertical_slash_gb300.pipeline import dense_causal_flops, flop_counts  # noqa: E402


def test_flop_counts_closed_form():
    # two heads: query-major slash tiles / bar chunks, key-major slash / bar units
    counts = np.array([[[3, 1, 5, 2]], [[7, 0, 4, 0]]], dtype=np.int64).reshape(1, 2, 4)
    d = 128
    f = flop_counts(counts, d)
    unit = 128 * 64
    q_units, k_units = 3 + 1 + 7 + 0, 5 + 2 + 4 + 0
    assert f["units"] == [10.0, 1.0, 9.0, 2.0]
    assert f["fwd_executed"] == pytest.approx(4 * q_units * unit * d)
    assert f["bwd_executed"] == pytest.approx(10 * q_units * unit * d)
    assert f["fwd_issued"] == f["fwd_executed"]
    # dQ: three GEMMs per query-major unit; dK / dV: four per key-major unit
    assert f["bwd_issued"] == pytest.approx((6 * q_units + 8 * k_units) * unit * d)


def test_dense_causal_flops_headline_shape():
    # one Qwen2.5-3B-shaped layer at 128K tokens: 16 query heads, d = 128
    f = dense_causal_flops(1, 131072, 16, 128)
    area = 16 * 131072 * 131073 / 2
    assert f["fwd"] == pytest.approx(4 * 128 * area)
    assert f["bwd"] == pytest.approx(2.5 * f["fwd"])
    assert f["fwd"] == pytest.approx(7.04e13, rel=1e-3)


def test_full_cover_credits_the_causal_tiles_plus_their_masked_halves():
    # a full causal cover of a 1K sequence by 128 x 64 query-major units
    # (T = 8 row tiles; tile t covers keys [0, 128 t + 127] in 2 t + 2 units)
    # is the dense causal area plus the masked upper halves of the diagonal tiles
    N, d, T = 1024, 64, 8
    units = sum(2 * t + 2 for t in range(T))
    counts = np.array([units, 0, 0, 0], dtype=np.int64).reshape(1, 1, 4)
    f = flop_counts(counts, d)
    dense = dense_causal_flops(1, N, 1, d)
    cover = units * 128 * 64
    assert cover == N * (N + 1) // 2 + T * (128 * 127 // 2)  # each diagonal 128 x 128 tile masks 128 * 127 / 2
    assert f["fwd_executed"] == pytest.approx(4.0 * cover * d)
    assert f["fwd_executed"] > dense["fwd"]


def _bench():
    import bench

    return bench


def test_host_cover_units_match_the_cover_definition():
    # the benchmark's host model of the query-major cover (used to put the CPU
    # oracle on the GPU line's accounting) against the brute-force greedy cover
    from test_cover import greedy_starts

    rng = np.random.default_rng(5)
    for N in (1024, 1088, 2048):
        for k in (1, 7, 60, 300):
            offs = np.sort(rng.choice(N, size=k, replace=False)).astype(np.int32)
            cols = np.sort(rng.choice(N, size=min(k, 130), replace=False)).astype(np.int32)
            starts = np.array(greedy_starts(offs, N))
            T = (N + 127) // 128
            want_slash = sum(int((starts <= 128 * t + 127).sum()) for t in range(T))
            want_bar = sum(int((cols[::64] <= 128 * t + 127).sum()) for t in range(T))
            got = _bench().query_cover_units(cols[None, None], offs[None, None], N)
            assert got.tolist() == [[[want_slash, want_bar]]], (N, k)


def test_host_cover_units_of_every_offset_is_the_causal_tiling():
    N = 1024
    got = _bench().query_cover_units(np.array([[[0]]], np.int32), np.arange(N, dtype=np.int32)[None, None], N)
    assert got[0, 0, 0] == sum(2 * t + 2 for t in range(N // 128))


def test_mask_entries_closed_form_against_the_oracle():
    import oracle

    rng = np.random.default_rng(9)
    N, H, kv, ks = 512, 3, 40, 70
    iv = np.stack([np.sort(rng.choice(N, kv, replace=False)) for _ in range(H)])[None].astype(np.int32)
    is_ = np.stack([np.sort(rng.choice(N, ks, replace=False)) for _ in range(H)])[None].astype(np.int32)
    is_[0, 1, -5:] = -1  # a padded (top-p) list
    is_[0, 1, :-5] = np.sort(rng.choice(N, ks - 5, replace=False))
    z = np.zeros((1, N, H, 1))
    p = oracle.Problem(z, np.zeros((1, N, 1, 1)), np.zeros((1, N, 1, 1)), iv, is_, 1.0)
    got = _bench().mask_entries(iv, is_, N)
    for h in range(H):
        assert got[0, h] == int(oracle.mask_dense(p, 0, h).sum())
    assert got.sum() == oracle.mask_count(p)


def test_block_mask_entries_closed_form_against_the_oracle():
    import oracle

    rng = np.random.default_rng(10)
    N, H = 640, 3
    iv = np.stack([np.sort(rng.choice(N, 24, replace=False)) for _ in range(H)])[None].astype(np.int32)
    is_ = np.stack([np.sort(rng.choice(N, 5, replace=False)) for _ in range(H)])[None].astype(np.int32)
    is_[0, 2, :] = [0, 64, 65, 300, 639]  # offsets on and between block multiples
    iv[0, 1, -3:] = -1  # a padded list
    iv[0, 1, :-3] = np.sort(rng.choice(N, 21, replace=False))
    p = oracle.Problem(np.zeros((1, N, H, 1)), np.zeros((1, N, 1, 1)), np.zeros((1, N, 1, 1)), iv, is_, 1.0, block=True)
    got = _bench().block_mask_entries(iv, is_, N)
    for h in range(H):
        assert got[0, h] == int(oracle.mask_dense(p, 0, h).sum())
    # every offset selected: the whole causal area
    full = _bench().block_mask_entries(iv, np.arange(N, dtype=np.int32)[None, None].repeat(H, 1), N)
    assert (full == N * (N + 1) // 2).all()
