"""Pins for the oracle's block-level striping and merge_out_and_lse
(Algorithm 2): hand-worked and page-printed figures, permutation identities,
and the exactness of merging per-step partial results into the global one."""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")))


def test_stripes_per_worker_from_pages():
    g = GOLDEN["stripes_per_worker"]
    pos = oracle.stripe_positions(g["seq_len"], g["workers"], g["stripe_tokens"], 5)
    starts = pos[:: g["stripe_tokens"]]
    assert len(starts) == g["stripes_per_worker"]
    assert np.all(np.diff(pos.reshape(-1, g["stripe_tokens"]), axis=1) == 1)  # stripes are contiguous


def test_striping_worked_example():
    g = GOLDEN["striping_worked_example"]
    for r, ranges in g["worker_positions"].items():
        want = np.concatenate([np.arange(a, b) for a, b in ranges])
        np.testing.assert_array_equal(oracle.stripe_positions(g["N"], g["W"], g["stripe"], int(r)), want)


def test_causal_area_cases_from_pages():
    for S, area in GOLDEN["causal_diagonal_block_area"]["cases"]:
        rng = np.random.default_rng(S)
        x = rng.standard_normal((1, S, 1, 4))
        p = oracle.Problem(x, x, x, np.zeros((1, 1, 1), np.int32), np.arange(S, dtype=np.int32)[None, None], 0.5)
        assert oracle.mask_count(p) == area


@pytest.mark.parametrize("W", [1, 2, 4])
def test_permute_roundtrip_and_positions(W):
    N, stripe = 512, 64
    x = np.random.default_rng(W).standard_normal((2, N, 3, 4))
    sh = oracle.striped_permute(x, W, stripe)
    np.testing.assert_array_equal(oracle.striped_permute(sh, W, stripe, inverse=True), x)
    for r in range(W):
        np.testing.assert_array_equal(sh[r], x[:, oracle.stripe_positions(N, W, stripe, r)])
    if W == 1:
        np.testing.assert_array_equal(sh[0], x)


def test_merge_closed_form():
    # merging the softmax over two disjoint key sets gives the softmax over the union
    rng = np.random.default_rng(3)
    s1, s2 = rng.standard_normal(5), rng.standard_normal(7)
    v1, v2 = rng.standard_normal((5, 3)), rng.standard_normal((7, 3))
    def part(s, v):
        l = np.log(np.sum(np.exp(s)))
        return np.exp(s - l) @ v, l
    o1, l1 = part(s1, v1)
    o2, l2 = part(s2, v2)
    o, l = oracle.merge(o1, l1, o2, l2)
    ow, lw = part(np.concatenate([s1, s2]), np.concatenate([v1, v2]))
    np.testing.assert_allclose(o, ow, atol=1e-14)
    assert l == pytest.approx(lw, abs=1e-14)
    o, l = oracle.merge(o1, l1, np.zeros(3), -np.inf)
    np.testing.assert_array_equal(o, o1)


def test_ring_steps_merge_to_global_rows():
    # worker 0 of W runs W steps against every KV shard (src = (0 - s) mod W)
    # with the global mask on global positions; merged, it equals the global
    # computation on worker 0's rows.
    N, W, stripe, Hq, Hkv, d = 512, 4, 64, 2, 1, 8
    rng = np.random.default_rng(11)
    q, k, v = rng.standard_normal((1, N, Hq, d)), rng.standard_normal((1, N, Hkv, d)), rng.standard_normal((1, N, Hkv, d))
    iv = np.sort(rng.choice(N, (1, Hq, 16), replace=True), -1)
    iv = np.stack([np.stack([np.sort(rng.choice(N, 16, replace=False)) for _ in range(Hq)])])
    is_ = np.stack([np.stack([np.sort(rng.choice(N, 24, replace=False)) for _ in range(Hq)])])
    scale = 1 / math.sqrt(d)
    glob = oracle.attention(oracle.Problem(q, k, v, iv, is_, scale))
    qpos = oracle.stripe_positions(N, W, stripe, 0)
    acc_o = np.zeros((len(qpos), Hq, d))
    acc_l = np.full((len(qpos), Hq), -np.inf)
    for s in range(W):
        src = (0 - s) % W
        kpos = oracle.stripe_positions(N, W, stripe, src)
        p = oracle.Problem(q[:, qpos], k[:, kpos], v[:, kpos], iv, is_, scale, qpos=qpos, kpos=kpos, n_global=N)
        part = oracle.attention(p)
        for n in range(len(qpos)):
            for h in range(Hq):
                acc_o[n, h], acc_l[n, h] = oracle.merge(acc_o[n, h], acc_l[n, h], part["o"][0, n, h],
                                                        part["lse"][0, h, n])
    np.testing.assert_allclose(acc_o, glob["o"][0, qpos], atol=1e-13)
    fin = np.isfinite(glob["lse"][0][:, qpos].T)
    np.testing.assert_array_equal(np.isfinite(acc_l), fin)
    np.testing.assert_allclose(acc_l[fin], glob["lse"][0][:, qpos].T[fin], atol=1e-13)
