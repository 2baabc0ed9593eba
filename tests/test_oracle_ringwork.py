"""Pins for the oracle's ring-layout work counts (MTraining, sections 2 and
4.2: Striped and ZigZag Ring Attention): a hand-worked example, the mask
area, and the pages' statement that both layouts balance full causal
attention across workers (exact for ZigZag)."""
import json
import os

import numpy as np
import pytest

import oracle
from vs_testutil import random_selection

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ring_work_n256_w2.json")


def _full(N, B=1, H=1):
    iv = np.zeros((B, H, 1), np.int32)  # column 0 is on every row's diagonal set too
    is_ = np.tile(np.arange(N, dtype=np.int32), (B, H, 1))
    return iv, is_


def test_hand_worked_example():
    g = json.load(open(GOLDEN))
    iv, is_ = _full(g["N"])
    for layout in ("striped", "zigzag"):
        got = oracle.ring_work(iv, is_, g["N"], g["W"], layout)
        assert got.tolist() == g[layout], layout


def test_owners():
    assert oracle.ring_owners(512, 2, "striped").reshape(-1, 64)[:, 0].tolist() == [0, 1] * 4
    assert oracle.ring_owners(512, 2, "zigzag").reshape(-1, 128)[:, 0].tolist() == [0, 1, 1, 0]
    z = oracle.ring_owners(1024, 4, "zigzag")
    assert all(np.count_nonzero(z == r) == 256 for r in range(4))


@pytest.mark.parametrize("layout", ["striped", "zigzag"])
def test_total_is_mask_area(layout):
    N, W = 1024, 4
    iv, is_ = random_selection(2, 3, N, 17, 40, 5)
    got = oracle.ring_work(iv, is_, N, W, layout)
    p = oracle.Problem(np.zeros((2, N, 3, 1)), np.zeros((2, N, 1, 1)), np.zeros((2, N, 1, 1)), iv, is_, 1.0)
    assert got.sum() == oracle.mask_count(p)


@pytest.mark.parametrize("N,W", [(512, 2), (1024, 4), (2048, 8)])
def test_zigzag_balances_full_causal(N, W):
    iv, is_ = _full(N)
    got = oracle.ring_work(iv, is_, N, W, "zigzag")
    tot = got.sum(1)
    assert (tot == tot[0]).all() and tot.sum() == N * (N + 1) // 2
    # striped is balanced too, up to its causal tail (the last worker holds
    # the latest block of every round of W blocks)
    st = oracle.ring_work(iv, is_, N, W, "striped").sum(1)
    assert st.max() / st.mean() < 1 + 2.0 * W / (N // 64)


def test_single_worker_is_everything():
    iv, is_ = random_selection(1, 2, 512, 9, 30, 7)
    for layout in ("striped", "zigzag"):
        got = oracle.ring_work(iv, is_, 512, 1, layout)
        p = oracle.Problem(np.zeros((1, 512, 2, 1)), np.zeros((1, 512, 1, 1)), np.zeros((1, 512, 1, 1)), iv, is_, 1.0)
        assert got.shape == (1, 1) and got[0, 0] == oracle.mask_count(p)


def test_zigzag_positions_hand_worked():
    # N = 16, W = 2: four chunks of 4 tokens; worker 0 holds chunks 0 and 3,
    # worker 1 chunks 1 and 2 (the mirrored pairs of the folded sequence)
    assert oracle.ring_positions(16, 2, 0, "zigzag").tolist() == [0, 1, 2, 3, 12, 13, 14, 15]
    assert oracle.ring_positions(16, 2, 1, "zigzag").tolist() == [4, 5, 6, 7, 8, 9, 10, 11]


@pytest.mark.parametrize("layout", ["striped", "zigzag"])
def test_ring_positions_are_the_owned_tokens_in_sequence_order(layout):
    N, W = 2048, 4
    own = oracle.ring_owners(N, W, layout)
    seen = np.zeros(N, np.int64)
    for r in range(W):
        pos = oracle.ring_positions(N, W, r, layout)
        np.testing.assert_array_equal(pos, np.nonzero(own == r)[0])  # ascending: local order = sequence order
        seen[pos] += 1
    assert np.all(seen == 1)


def test_ring_permute_moves_each_token_to_its_owner():
    N, W = 1024, 4
    x = np.arange(N, dtype=np.int64).reshape(1, N, 1, 1)
    for layout in ("striped", "zigzag"):
        y = oracle.ring_permute(x, W, layout)
        assert y.shape == (W, 1, N // W, 1, 1)
        own = oracle.ring_owners(N, W, layout)
        for r in range(W):
            assert np.all(own[y[r, 0, :, 0, 0]] == r)
    np.testing.assert_array_equal(oracle.ring_permute(x, W, "striped"), oracle.striped_permute(x, W, 64))
