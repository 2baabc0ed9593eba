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
