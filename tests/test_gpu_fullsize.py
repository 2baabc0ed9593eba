"""Parity at the full sizes of the named workloads, through the same buffers
and launches the benchmark times (``VSAttention`` / ``StripedWorker``), on
outputs the fp64 oracle computes one at a time:

* selection: the GPU's fp32 scores against the oracle's fp64 estimate
  (within 1e-4 of the largest score), the GPU's indices bit-exact under the
  replay rule (the oracle's top-k on the GPU's own scores), and every index
  on which the two selections differ inside the tolerance band of the k-th
  score;
* attention, on the oracle's own selection: O, LSE and dQ of 64 sampled
  query rows of every head (the first rows, which only the vertical bars
  reach, rows of the heaviest last query tile, and random rows) and dK / dV
  of 32 sampled keys of every KV head (the last keys of the sequence,
  vertical ones among them, keys in the middle that only slash lines reach,
  and vertical keys past the middle whose attending rows cross several of the
  key-major bar kernel's split pieces), with O / dQ / dK / dV relative L2
  <= 1e-2 over the sample (per-head values printed; each head's own sample
  below 3e-2) and LSE absolute <= 1e-3.

The oracle widens only the rows it needs: the query / dO rows of the sampled
rows and of every row that reaches a sampled key.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from vs_testutil import dev_bf16, host_f64, rel_l2

pytestmark = pytest.mark.gpu

TOL = 1e-2
SCORE_TOL = 1e-4


@pytest.fixture(scope="module")
def vs():
    import dynamic_vertical_slash_gb300 as m

    m.lib()
    return m


def _f64(bits):
    return synth.bf16_to_f32(bits).astype(np.float64)


def _oracle_scores(x, w):
    """Oracle estimate: only the last ``last_q`` query rows are read, so the
    rest of q is left as zeros (never widened)."""
    B, N, Hq, d = x["q"].shape
    q = np.zeros((B, N, Hq, d), np.float64)
    q[:, N - w.last_q:] = _f64(x["q"][:, N - w.last_q:])
    return oracle.estimate(q, _f64(x["k"]), w.last_q, w.scale)


def _check_selection(v_gpu, s_gpu, iv_gpu, is_gpu, v_ref, s_ref, iv_ref, is_ref, kv, ks):
    B, Hq, N = v_ref.shape
    for b in range(B):
        for h in range(Hq):
            for sc_g, sc_r, idx_g, idx_r, k in ((v_gpu, v_ref, iv_gpu, iv_ref, kv), (s_gpu, s_ref, is_gpu, is_ref, ks)):
                top = sc_r[b, h].max()
                assert np.max(np.abs(sc_g[b, h] - sc_r[b, h])) <= SCORE_TOL * top, (b, h)
                np.testing.assert_array_equal(oracle.topk(sc_g[b, h], k), idx_g[b, h])
                diff = np.setxor1d(idx_g[b, h], idx_r[b, h])
                if diff.size:
                    kth = np.sort(sc_r[b, h])[::-1][k - 1]
                    assert np.all(np.abs(sc_r[b, h][diff] - kth) <= 2 * SCORE_TOL * top), (b, h, diff)


def _sample_rows(N, rng, count=64):
    """The first rows, rows of the last 128-row tile (the heaviest), random rows."""
    first = np.arange(8)
    last = np.sort(rng.choice(np.arange(N - 128, N), 16, replace=False))
    mid = rng.choice(np.arange(8, N - 128), count - 24, replace=False)
    return np.unique(np.concatenate([first, last, mid]))


def _rows_reaching(m, ivh, ish, N):
    """Every row n >= m whose mask holds key m in one of the given heads."""
    rows = set()
    for iv_row, is_row in zip(ivh, ish):
        if m in set(iv_row.tolist()):
            rows.update(range(m, N))
        rows.update(int(m + o) for o in is_row if m + o < N)
    return rows


def _sample_keys(b, hk, g, iv, is_, N, rng, dense):
    """32 keys of KV head hk: the last ones (vertical ones preferred); unless
    the mask is dense, also mid-sequence keys no vertical list holds (only
    slash lines reach them) and vertical keys in [5N/8, 3N/4), whose
    attending rows span more than one 16384-row piece of the key-major bar
    kernel."""
    tail = 128 if dense else 2048
    ivh = iv[b, hk * g:(hk + 1) * g]
    vert = sorted({int(m) for m in ivh.ravel() if m >= N - tail})
    keys = set(vert[-8:])
    if not dense:
        held = set(ivh.ravel().tolist())
        slash_only = [int(m) for m in rng.permutation(np.arange(N // 4, 3 * N // 4))[:64] if int(m) not in held]
        keys |= set(slash_only[:4])
        mid_vert = sorted({int(m) for m in ivh.ravel() if 5 * N // 8 <= m < 3 * N // 4})
        if mid_vert:
            keys |= set(rng.choice(mid_vert, min(4, len(mid_vert)), replace=False).tolist())
    for m in rng.permutation(np.arange(N - tail, N)):
        if len(keys) >= 32:
            break
        keys.add(int(m))
    return sorted(keys)


HEAD_TOL = 3e-2  # a single head's small sample: only a gross per-head fault exceeds it


def _per_head(name, got, ref, heads):
    """Relative L2 of every head's sample (heads: the head of each sample
    row), reported with the worst; the tolerance of the comparison is the
    whole sample's (asserted by the caller), a head's own sample only has to
    stay below HEAD_TOL."""
    errs = {int(h): rel_l2(got[heads == h], ref[heads == h]) for h in np.unique(heads)}
    worst = max(errs, key=errs.get)
    print("%s: worst head %d rel-L2 %.3g, sample rel-L2 %.3g; per head %s" % (
        name, worst, errs[worst], rel_l2(got, ref), {h: round(e, 4) for h, e in errs.items()}))
    assert errs[worst] <= HEAD_TOL, (name, errs)


def _compare_rows(p, rows_bhn, o_gpu, lse_gpu, dq_gpu):
    o_ref, lse_ref, dq_ref = oracle.rows(p, rows_bhn)
    assert rel_l2(o_gpu, o_ref) <= TOL
    assert rel_l2(dq_gpu, dq_ref) <= TOL
    _per_head("O", o_gpu, o_ref, rows_bhn[:, 1])
    _per_head("dQ", dq_gpu, dq_ref, rows_bhn[:, 1])
    fin = np.isfinite(lse_ref)
    np.testing.assert_array_equal(np.isfinite(lse_gpu), fin)
    assert np.max(np.abs(lse_gpu[fin] - lse_ref[fin]), initial=0.0) <= 1e-3


@pytest.mark.parametrize("name", ["qwen3b-32k", "qwen3b-128k", "batch4-64k", "dense-64k"])
def test_fullsize_sampled_parity(vs, name):
    w = synth.workloads()[name]
    x = synth.make_batch(w)
    B, N, Hq, Hkv, d, g = w.B, w.N, w.Hq, w.Hkv, w.d, w.Hq // w.Hkv
    dense = w.ks >= N
    q, k, v, do = (dev_bf16(x[n]) for n in ("q", "k", "v", "dout"))
    att = vs.VSAttention(B, N, Hq, Hkv, d, w.kv, w.ks, last_q=w.last_q, scale=w.scale)

    # ---- selection: the pipeline's own estimator against the oracle's
    att.forward(q, k, v)
    torch.cuda.synchronize()
    att.check()
    v_gpu, s_gpu = att.v_score.cpu().numpy(), att.s_score.cpu().numpy()
    iv_gpu, is_gpu = att.v_idx.cpu().numpy(), att.s_idx.cpu().numpy()
    v_ref, s_ref = _oracle_scores(x, w)
    iv, is_ = oracle.select(v_ref, s_ref, w.kv, w.ks)
    _check_selection(v_gpu, s_gpu, iv_gpu, is_gpu, v_ref, s_ref, iv, is_, w.kv, w.ks)

    # ---- attention on the oracle's selection, same buffers and launches
    _attention_sampled(w, x, att, iv, is_, q, k, v, do, dense)


def _attention_sampled(w, x, att, iv, is_, q, k, v, do, dense):
    """Forward and backward of `att` on the selection (iv, is_) against the
    oracle on sampled rows and keys."""
    B, N, Hq, Hkv, g = w.B, w.N, w.Hq, w.Hkv, w.Hq // w.Hkv
    att.forward(q, k, v, selection=(torch.from_numpy(iv).cuda(), torch.from_numpy(is_).cuda()))
    dq, dk, dv = att.backward(do)
    torch.cuda.synchronize()
    att.check()
    o_h, lse_h = host_f64(att.o), att.lse.cpu().numpy().astype(np.float64)
    dq_h, dk_h, dv_h = host_f64(dq), host_f64(dk), host_f64(dv)
    kf, vf = _f64(x["k"]), _f64(x["v"])
    rng = np.random.default_rng(99)
    for b in range(B):
        rows = _sample_rows(N, rng)
        keys = {hk: _sample_keys(b, hk, g, iv, is_, N, rng, dense) for hk in range(Hkv)}
        need = set(rows.tolist())
        for hk, ks_ in keys.items():
            for m in ks_:
                need |= _rows_reaching(m, iv[b, hk * g:(hk + 1) * g], is_[b, hk * g:(hk + 1) * g], N)
        pos = np.array(sorted(need), np.int64)
        loc = {int(n): i for i, n in enumerate(pos)}
        p = oracle.Problem(_f64(x["q"][b:b + 1, pos]), kf[b:b + 1], vf[b:b + 1], iv[b:b + 1], is_[b:b + 1],
                           w.scale, dout=_f64(x["dout"][b:b + 1, pos]), qpos=pos, n_global=N)
        rb = np.array([(0, h, loc[int(n)]) for h in range(Hq) for n in rows], np.int32)
        _compare_rows(p, rb, np.stack([o_h[b, n, h] for h in range(Hq) for n in rows]),
                      np.array([lse_h[b, h, n] for h in range(Hq) for n in rows]),
                      np.stack([dq_h[b, n, h] for h in range(Hq) for n in rows]))
        kb = np.array([(0, hk, m) for hk in range(Hkv) for m in keys[hk]], np.int32)
        dk_ref, dv_ref = oracle.keys(p, kb)
        got_k = np.stack([dk_h[b, m, hk] for hk in range(Hkv) for m in keys[hk]])
        got_v = np.stack([dv_h[b, m, hk] for hk in range(Hkv) for m in keys[hk]])
        assert rel_l2(got_k, dk_ref) <= TOL
        assert rel_l2(got_v, dv_ref) <= TOL
        _per_head("dK", got_k, dk_ref, kb[:, 1])
        _per_head("dV", got_v, dv_ref, kb[:, 1])


def test_fullsize_packed_group_selection_sampled_parity(vs):
    """The per-KV-group selection with the group's heads packed into the
    query-major tiles (VSAttention(shared=True, packed=True)) at 128K: the
    selection replays bit-exactly from the GPU's own fp32 group sums, and the
    attention on the oracle's fp64 group selection matches on sampled rows
    and keys."""
    w = synth.workloads()["qwen3b-128k"]
    x = synth.make_batch(w)
    B, N, Hq, Hkv, d, g = w.B, w.N, w.Hq, w.Hkv, w.d, w.Hq // w.Hkv
    q, k, v, do = (dev_bf16(x[n]) for n in ("q", "k", "v", "dout"))
    att = vs.VSAttention(B, N, Hq, Hkv, d, w.kv, w.ks, last_q=w.last_q, scale=w.scale, shared=True, packed=True)
    att.forward(q, k, v)
    torch.cuda.synchronize()
    att.check()
    v_gpu, s_gpu = att.v_score.cpu().numpy(), att.s_score.cpu().numpy()
    iv_r, is_r = oracle.select_group(v_gpu, s_gpu, w.kv, w.ks, g, dtype=np.float32)
    np.testing.assert_array_equal(att.v_idx.cpu().numpy(), iv_r)
    np.testing.assert_array_equal(att.s_idx.cpu().numpy(), is_r)
    v_ref, s_ref = _oracle_scores(x, w)
    iv, is_ = oracle.select_group(v_ref, s_ref, w.kv, w.ks, g)
    _attention_sampled(w, x, att, iv, is_, q, k, v, do, False)


def test_fullsize_striped_ring_sampled_parity(vs):
    """Worker 0 of the 8-worker striped ring at 524288 global tokens, in the
    benchmark's launches: global selection, one index per ring step, merged
    forward, accumulated dQ and per-source dK / dV, against the oracle's
    global computation on worker 0's rows."""
    w = synth.workloads()["qwen3b-512k-striped8"]
    x = synth.make_batch(w)
    B, N, Hq, Hkv, d, W, g = w.B, w.N, w.Hq, w.Hkv, w.d, w.world, w.Hq // w.Hkv
    q, k, v, do = (dev_bf16(x[n]) for n in ("q", "k", "v", "dout"))
    q0 = vs.striped_permute(q, W, w.stripe, only_rank=0)
    do0 = vs.striped_permute(do, W, w.stripe, only_rank=0)
    ksh, vsh = vs.striped_permute(k, W, w.stripe), vs.striped_permute(v, W, w.stripe)
    del do
    wk = vs.StripedWorker(B, N, Hq, Hkv, d, w.kv, w.ks, W, rank=0, stripe=w.stripe, last_q=w.last_q, scale=w.scale)
    wk.select(q, k)
    torch.cuda.synchronize()
    v_ref, s_ref = _oracle_scores(x, w)
    iv, is_ = oracle.select(v_ref, s_ref, w.kv, w.ks)
    _check_selection(wk.v_score.cpu().numpy(), wk.s_score.cpu().numpy(), wk.v_idx.cpu().numpy(),
                     wk.s_idx.cpu().numpy(), v_ref, s_ref, iv, is_, w.kv, w.ks)
    wk.v_idx.copy_(torch.from_numpy(iv))
    wk.s_idx.copy_(torch.from_numpy(is_))
    wk.build_index(q0, ksh)
    wk.forward(q0, ksh, vsh)
    dq, dk, dv = wk.backward(do0)
    torch.cuda.synchronize()
    wk.check()
    c = wk.counts()
    assert c.shape == (W, B, Hq, 4) and np.all(c[:, :, :, 0] > 0)

    pos0 = oracle.stripe_positions(N, W, w.stripe, 0)
    rng = np.random.default_rng(7)
    li = np.unique(np.concatenate([[0, 1, len(pos0) - 1], rng.choice(len(pos0), 5, replace=False)]))
    tail = pos0[pos0 >= N - 2048]
    need = np.unique(np.concatenate([pos0[li], tail]))
    p = oracle.Problem(_f64(x["q"][:, need]), _f64(x["k"]), _f64(x["v"]), iv, is_, w.scale,
                       dout=_f64(x["dout"][:, need]), qpos=need, n_global=N)
    loc = {int(n): i for i, n in enumerate(need)}
    o_h, lse_h, dq_h = host_f64(wk.o), wk.lse.cpu().numpy().astype(np.float64), host_f64(dq)
    rb = np.array([(0, h, loc[int(pos0[i])]) for h in range(Hq) for i in li], np.int32)
    _compare_rows(p, rb, np.stack([o_h[0, i, h] for h in range(Hq) for i in li]),
                  np.array([lse_h[0, h, i] for h in range(Hq) for i in li]),
                  np.stack([dq_h[0, i, h] for h in range(Hq) for i in li]))
    # dK / dV of the last keys of each source shard, from worker 0's rows
    # (rows >= N - 2048 are all in the problem, so every row reaching a key
    # m >= N - 2048 is present)
    dk_h, dv_h = host_f64(dk), host_f64(dv)
    got_k, got_v, kb = [], [], []
    for src in range(W):
        kpos = oracle.stripe_positions(N, W, w.stripe, src)
        for j in np.nonzero(kpos >= N - 2048)[0][-2:]:
            for hk in range(Hkv):
                kb.append((0, hk, int(kpos[j])))
                got_k.append(dk_h[src, 0, j, hk])
                got_v.append(dv_h[src, 0, j, hk])
    dk_ref, dv_ref = oracle.keys(p, np.array(kb, np.int32))
    assert rel_l2(np.stack(got_k), dk_ref) <= TOL
    assert rel_l2(np.stack(got_v), dv_ref) <= TOL
