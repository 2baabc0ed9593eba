"""Pins for the oracle's per-KV-group shared selection: one head per group
is the per-head selection, identical heads select what one head selects, and
a brute-force sort of the summed scores."""
import numpy as np

import oracle


def test_one_head_per_group_is_per_head():
    rng = np.random.default_rng(1)
    v, s = rng.random((2, 4, 300)), rng.random((2, 4, 300))
    a = oracle.select_group(v, s, 20, 30, 1)
    b = oracle.select(v, s, 20, 30)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_identical_heads():
    rng = np.random.default_rng(2)
    v1, s1 = rng.random((1, 1, 500)), rng.random((1, 1, 500))
    v, s = np.repeat(v1, 4, 1), np.repeat(s1, 4, 1)  # 4 identical heads, one group
    iv, is_ = oracle.select_group(v, s, 17, 9, 4)
    r = oracle.select(v1, s1, 17, 9)
    for h in range(4):
        np.testing.assert_array_equal(iv[0, h], r[0][0, 0])
        np.testing.assert_array_equal(is_[0, h], r[1][0, 0])


def test_brute_force_sum_and_sharing():
    rng = np.random.default_rng(3)
    v = rng.random((1, 6, 200))
    s = rng.random((1, 6, 200))
    iv, is_ = oracle.select_group(v, s, 12, 25, 3)  # 2 groups of 3 heads
    for hk in range(2):
        tot = v[0, 3 * hk:3 * hk + 3].sum(0)
        want = np.sort(np.argsort(-tot, kind="stable")[:12])
        for h in range(3 * hk, 3 * hk + 3):
            np.testing.assert_array_equal(iv[0, h], want)
            np.testing.assert_array_equal(is_[0, h], is_[0, 3 * hk])
