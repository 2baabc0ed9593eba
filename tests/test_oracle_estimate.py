"""Pins for the oracle's estimator (Algorithm 1, observation window) and
top-k selection: closed forms, a library softmax, brute force and planted
ties -- none of them re-use the oracle's own code."""
import math

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_rows_of_window_sum_to_one():
    # each softmax row sums to 1 (Theorem 3.1's attention-score definition),
    # so sum_m v[m] = sum_o s[o] = last_q
    B, N, Hq, Hkv, d, lq = 2, 200, 4, 2, 16, 64
    q, k = _rand((B, N, Hq, d), 1), _rand((B, N, Hkv, d), 2)
    v, s = oracle.estimate(q, k, lq, 1 / math.sqrt(d))
    np.testing.assert_allclose(v.sum(-1), lq, rtol=0, atol=1e-11)
    np.testing.assert_allclose(s.sum(-1), lq, rtol=0, atol=1e-11)
    assert (v >= 0).all() and (s >= 0).all()


def test_zero_keys_closed_form():
    # K = 0: every causal logit is 0, so A_hat[i, m] = 1 / (n_i + 1)
    N, d, lq = 300, 8, 64
    q = _rand((1, N, 1, d), 3)
    k = np.zeros((1, N, 1, d))
    v, s = oracle.estimate(q, k, lq, 0.3)
    n = np.arange(N - lq, N)
    want = np.array([np.sum(1.0 / (n[n >= m] + 1)) for m in range(N)])
    np.testing.assert_allclose(v[0, 0], want, rtol=1e-13, atol=0)
    np.testing.assert_allclose(s[0, 0], want, rtol=1e-13, atol=0)


def test_planted_diagonal_closed_form():
    # q_{n_i} = L e_i; the key at m_i = n_i - o* is e_i; every other key is 0.
    # Row i has one logit a = scale * L at m_i and zeros elsewhere, so
    #   s[o*] = sum_i e^a / (e^a + n_i)
    #   s[o]  = sum_{i: n_i >= o} 1 / (e^a + n_i)            (o != o*)
    #   v[m_i] = e^a/(e^a+n_i) + sum_{j != i, n_j >= m_i} 1/(e^a + n_j)
    N, lq, ostar, L = 400, 64, 100, 6.0
    d = lq
    scale = 1 / math.sqrt(d)
    q = np.zeros((1, N, 1, d))
    k = np.zeros((1, N, 1, d))
    n = np.arange(N - lq, N)
    for i in range(lq):
        q[0, n[i], 0, i] = L
        k[0, n[i] - ostar, 0, i] = 1.0
    v, s = oracle.estimate(q, k, lq, scale)
    ea = math.exp(scale * L)
    want_s = np.array([np.sum(1.0 / (ea + n[n >= o])) for o in range(N)])
    want_s[ostar] = np.sum(ea / (ea + n))
    np.testing.assert_allclose(s[0, 0], want_s, rtol=1e-12)
    for i in (0, 17, lq - 1):
        m = n[i] - ostar
        others = [j for j in range(lq) if j != i and n[j] >= m]
        want_v = ea / (ea + n[i]) + sum(1.0 / (ea + n[j]) for j in others)
        assert v[0, 0, m] == pytest.approx(want_v, rel=1e-12)
    # the selection picks the planted diagonal first
    assert oracle.topk(s[0, 0], 1)[0] == ostar


def test_estimate_matches_library_softmax():
    B, N, Hq, Hkv, d, lq = 1, 160, 4, 2, 32, 64
    q, k = _rand((B, N, Hq, d), 5), _rand((B, N, Hkv, d), 6)
    scale = 1 / math.sqrt(d)
    v, s = oracle.estimate(q, k, lq, scale)
    g = Hq // Hkv
    for h in range(Hq):
        Q = torch.tensor(q[0, N - lq:, h])
        K = torch.tensor(k[0, :, h // g])
        logits = Q @ K.T * scale
        n = torch.arange(N - lq, N)[:, None]
        m = torch.arange(N)[None, :]
        A = torch.softmax(logits.masked_fill(m > n, float("-inf")), dim=-1).numpy()
        np.testing.assert_allclose(v[0, h], A.sum(0), rtol=1e-12, atol=1e-15)
        s_want = np.zeros(N)
        for i in range(lq):
            ni = N - lq + i
            s_want[: ni + 1] += A[i, ni::-1][: ni + 1]
        np.testing.assert_allclose(s[0, h], s_want, rtol=1e-12, atol=1e-15)


# ------------------------------------------------------------------ top-k
def _brute_topk(score, k):
    order = np.lexsort((np.arange(score.size), -score))  # score desc, index asc
    return np.sort(order[:k])


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 3000))
    score = rng.integers(0, 7, n).astype(np.float64) * 0.25  # many exact ties
    for k in {1, n // 3 + 1, n}:
        np.testing.assert_array_equal(oracle.topk(score, k), _brute_topk(score, k))


def test_topk_ties_go_to_lowest_index():
    np.testing.assert_array_equal(oracle.topk(np.ones(100), 7), np.arange(7))
    s = np.zeros(50)
    s[[3, 9, 40]] = 2.0
    s[[5, 6, 30]] = 1.0
    np.testing.assert_array_equal(oracle.topk(s, 4), [3, 5, 9, 40])


def test_topk_float32_replay_is_exact():
    rng = np.random.default_rng(9)
    s32 = rng.random(5000).astype(np.float32)
    s32[100:200] = s32[100]  # ties at float32 precision
    got = oracle.topk(s32, 300)
    np.testing.assert_array_equal(got, _brute_topk(s32.astype(np.float64), 300))


def test_planted_columns_are_selected():
    import synth

    w = synth.small_workload(N=1024, Hq=2, Hkv=1, d=64, kv=8, ks=8, seed=1, n_out=8)
    x = synth.make_batch(w, with_dout=False)
    q, k = synth.bf16_to_f32(x["q"]), synth.bf16_to_f32(x["k"])
    v, s = oracle.estimate(q, k, 64, w.scale)
    iv, _ = oracle.select(v, s, 8, 8)
    for h in range(2):
        np.testing.assert_array_equal(iv[0, h], x["planted_cols"][0][0])
