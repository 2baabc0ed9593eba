"""Pins for the oracle's top-p budgets (Algorithm 1 of MTraining, the ``topp``
and ``Pool`` lines; section 4.1 (i), online budget approximation): brute
force over subsets, closed forms, invariants, and the padding rule of the
mask (entries -1 pad a list whose budget is below its capacity).  None of
them re-use the oracle's own sort-and-cumsum."""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle

UNIT = 2 ** oracle.MASS_UNIT_LOG2


def _brute_budget(units, p):
    """Smallest k whose best k-subset (exhaustive) reaches ceil(p * T)."""
    units = [int(x) for x in units]
    T = sum(units)
    t = math.ceil(float(p) * float(T))
    for k in range(len(units) + 1):
        best = max((sum(c) for c in itertools.combinations(units, k)), default=0)
        if best >= t:
            return k
    return len(units)


@pytest.mark.parametrize("seed", range(12))
def test_budget_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 10))
    x = rng.random(n) ** 3  # skewed masses, many near-ties in sum
    if seed % 3 == 0:
        x[rng.integers(0, n)] = x.max()  # exact ties
    u = oracle.mass_units(x)
    for p in (0.0, 0.1, 0.37, 0.5, 0.9, 0.999, 1.0):
        assert oracle.topp_budget(u, p) == _brute_budget(u, p), (p, x)


@pytest.mark.parametrize("n", [1, 7, 64, 1000])
@pytest.mark.parametrize("p", [0.25, 0.375, 0.5, 0.75, 1.0])
def test_uniform_closed_form(n, p):
    # equal scores: the k largest carry k / n of the mass, so k = ceil(p n)
    # (dyadic p keeps p * T exact)
    u = oracle.mass_units(np.full(n, 0.125))
    assert oracle.topp_budget(u, p) == math.ceil(Fraction(p) * n)


def test_target_is_one_rounded_double_product():
    # t = ceil(fl(p * T)): a hundred one-unit scores with p = 0.07 give
    # fl(0.07 * 100) = 7.000000000000001, so the budget is 8, not 7; with 100
    # equal scores fl(0.9 * T) rounds to exactly 90 T / 100, so 90
    assert 0.07 * 100 > 7
    assert oracle.topp_budget(oracle.mass_units(np.full(100, 2.0 ** -40)), 0.07) == 8
    u = oracle.mass_units(np.full(100, 0.5))
    assert oracle.topp_budget(u, 0.9) == 90
    assert oracle.topp_budget(u, 0.89) == 89


def test_dominant_score_and_extremes():
    x = np.full(500, 1e-3)
    x[137] = 60.0  # holds > 99% of the mass
    u = oracle.mass_units(x)
    assert oracle.topp_budget(u, 0.99) == 1
    assert oracle.topp_budget(u, 0.0) == 0
    # p = 1: every entry with a positive unit count
    x[:10] = 0.0
    x[10:20] = 2.0 ** -45  # below one unit
    assert oracle.topp_budget(oracle.mass_units(x), 1.0) == 480
    assert oracle.topp_budget(oracle.mass_units(np.zeros(8)), 0.5) == 0


def test_geometric_closed_form():
    # x_i = 2^-i: the k largest sum to 2 - 2^(1-k) (times the scale), exact
    # in units; k = smallest with that >= ceil(p T)
    n = 30
    x = 2.0 ** -np.arange(n)
    u = oracle.mass_units(x)
    T = int(u.sum())
    assert T == sum(UNIT >> i for i in range(n))
    for p in (0.5, 0.75, 0.9, 0.99, 0.999999):
        t = math.ceil(p * T)
        want = next(k for k in range(1, n + 1) if sum(UNIT >> i for i in range(k)) >= t)
        assert oracle.topp_budget(u, p) == want


def test_budget_invariants():
    rng = np.random.default_rng(5)
    x = rng.random(777)
    u = oracle.mass_units(x)
    for p in (0.3, 0.8):
        k = oracle.topp_budget(u, p)
        assert oracle.topp_budget(u[rng.permutation(u.size)], p) == k
        # monotone in p
        assert oracle.topp_budget(u, p + 0.05) >= k
    # doubling every score doubles every unit count: same budgets
    x2 = np.round(x * 2 ** 20) / 2 ** 20  # multiples of 2^-20: floor is exact
    assert np.array_equal(oracle.mass_units(2 * x2), 2 * oracle.mass_units(x2))
    assert oracle.topp_budget(oracle.mass_units(2 * x2), 0.6) == oracle.topp_budget(oracle.mass_units(x2), 0.6)


def test_mass_units_floor():
    x = np.array([0.0, 1.0, 2.0 ** -40, 2.0 ** -41, 0.75 + 2.0 ** -41, 64.0], np.float32)
    assert oracle.mass_units(x).tolist() == [0, UNIT, 1, 0, 3 * UNIT // 4, 64 * UNIT]


def test_pool_closed_form():
    u = np.arange(200, dtype=np.int64)
    got = oracle.pool(u, 64)
    # blocks [0,64), [64,128), [128,192), [192,200): arithmetic series
    want = [sum(range(a, min(a + 64, 200))) for a in (0, 64, 128, 192)]
    assert got.tolist() == want


def test_select_topp_slash_budget_counts_pooled_blocks():
    # all slash mass on offsets 70..80 (one 64-block): one block carries it all
    N = 512
    v = np.full((1, 1, N), 1.0 / N)
    s = np.zeros((1, 1, N))
    s[0, 0, 70:81] = 1.0
    iv, is_, kv, ks = oracle.select_topp(v, s, 0.5, 0.9, 300, 200)
    assert ks[0, 0] == 64 and kv[0, 0] == 256
    # the slash list: the 11 positive offsets first in score order (equal,
    # so lowest index first), then the lowest zero-score offsets
    got = is_[0, 0, :64]
    assert set(range(70, 81)) <= set(got.tolist())
    assert (is_[0, 0, 64:] == -1).all()
    assert np.all(np.diff(got) > 0)
    # mass split over two blocks: two blocks at ps above one block's share
    s[0, 0, 130:140] = 1.0
    _, _, _, ks2 = oracle.select_topp(v, s, 0.5, 0.6, 300, 200)
    assert ks2[0, 0] == 128


def test_select_topp_caps_and_padding():
    rng = np.random.default_rng(2)
    v = rng.random((2, 3, 256))
    s = rng.random((2, 3, 256))
    iv, is_, kv, ks = oracle.select_topp(v, s, 0.99, 1.0, 40, 100)
    assert (kv == 40).all() and (ks == 100).all()  # both capped
    iv, is_, kv, ks = oracle.select_topp(v, s, 0.3, 0.2, 256, 256)
    for b in range(2):
        for h in range(3):
            k = kv[b, h]
            head = iv[b, h, :k]
            assert (iv[b, h, k:] == -1).all() and np.all(np.diff(head) > 0)
            # minimality, checked by brute rule on the scores: the chosen set
            # reaches the target, one fewer of the largest does not
            u = oracle.mass_units(v[b, h])
            t = math.ceil(0.3 * float(u.sum()))
            assert u[head].sum() >= t
            assert np.sort(u)[::-1][:k - 1].sum() < t
            assert ks[b, h] % 64 == 0


def test_padded_lists_give_the_unpadded_mask():
    # the mask ignores -1 entries: a list padded to a larger capacity encodes
    # the same M as the list alone
    rng = np.random.default_rng(9)
    B, N, Hq, Hkv, d = 1, 300, 2, 1, 8
    q, k, v = rng.standard_normal((B, N, Hq, d)), rng.standard_normal((B, N, Hkv, d)), rng.standard_normal(
        (B, N, Hkv, d))
    iv = np.sort(rng.choice(N, (B, Hq, 5), replace=False), -1).astype(np.int32)
    is_ = np.sort(rng.choice(N, (B, Hq, 7), replace=False), -1).astype(np.int32)
    ivp = np.concatenate([iv, np.full((B, Hq, 11), -1, np.int32)], -1)
    isp = np.concatenate([is_, np.full((B, Hq, 3), -1, np.int32)], -1)
    p0 = oracle.Problem(q, k, v, iv, is_, 0.3)
    p1 = oracle.Problem(q, k, v, ivp, isp, 0.3)
    assert oracle.mask_count(p0) == oracle.mask_count(p1)
    for h in range(Hq):
        assert np.array_equal(oracle.mask_dense(p0, 0, h), oracle.mask_dense(p1, 0, h))
    # an all-padding head is the empty mask
    empty = oracle.Problem(q, k, v, np.full((B, Hq, 4), -1, np.int32), np.full((B, Hq, 4), -1, np.int32), 0.3)
    assert oracle.mask_count(empty) == 0
    o, lse, _ = oracle.rows(empty, np.array([[0, 0, 5], [0, 1, 299]]))
    assert np.all(o == 0) and np.all(np.isneginf(lse))
