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
