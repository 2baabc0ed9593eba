"""Top-p budgets on the GPU (Algorithm 1 of MTraining, `topp` and `Pool`)
against the oracle, through the C ABI.

Budgets and lists are integers decided from sums of scores; both sides take
the decision in the same exact precision (integer mass units of 2^-40 of a
score, target ceil(p * T)), so on the same fp32 scores they must agree bit
for bit.  Scores come from the seeded generator (``synth.score_lists``) or,
for the estimator, the GPU's own fp32 scores are replayed through the
oracle's selection (the replay rule of the fixed-budget estimator tests);
attention then runs on the oracle's own top-p selection from its fp64
estimate, padded lists and all.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from vs_testutil import Arena, dev_bf16, host_f64, make_inputs, rel_l2

pytestmark = pytest.mark.gpu

VS_ERR_INDEX, VS_ERR_SHAPE, VS_ERR_SCORE = 4, 2, 7


@pytest.fixture(scope="module")
def vs():
    import dynamic_vertical_slash_gb300 as m

    m.lib()
    return m


def _select(vs, v, s, pv, ps, kv_max, ks_max):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    out = vs.vs_select_topp(torch.from_numpy(v).cuda(), torch.from_numpy(s).cuda(), pv, ps, kv_max, ks_max, ws=ws)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in out], vs.vs_check_status(ws)


def _assert_same(got, ref):
    for g, r, name in zip(got, ref, ("iv", "is", "kv", "ks")):
        np.testing.assert_array_equal(g, r, err_msg=name)


@pytest.mark.parametrize("B,H,N,pv,ps,kv_max,ks_max,seed", [
    (2, 3, 4096, 0.9, 0.9, 4096, 4096, 1),
    (2, 3, 4096, 0.5, 0.5, 300, 4096, 2),      # kv capped for some heads
    (1, 4, 1088, 0.95, 0.99, 1088, 1000, 3),   # N not a multiple of 128; ks capped
    (1, 2, 64, 0.7, 0.7, 64, 64, 4),           # one pooled block
    (3, 2, 8192, 0.999, 0.3, 8192, 8192, 5),
])
def test_select_topp_matches_oracle(vs, B, H, N, pv, ps, kv_max, ks_max, seed):
    v, s = synth.score_lists(B, H, N, seed)
    got, st = _select(vs, v, s, pv, ps, kv_max, ks_max)
    assert st == 0
    _assert_same(got, oracle.select_topp(v, s, pv, ps, kv_max, ks_max))


def test_select_topp_full_size(vs):
    # 128K keys, 16 heads (the Qwen2.5-3B 128K shape): uncapped and capped
    v, s = synth.score_lists(1, 16, 131072, 7)
    for pv, ps, cap in ((0.6, 0.7, 131072), (0.9, 0.9, 2048)):
        got, st = _select(vs, v, s, pv, ps, cap, cap)
        assert st == 0
        _assert_same(got, oracle.select_topp(v, s, pv, ps, cap, cap))


def test_select_topp_largest_supported_n(vs):
    N = 1572864
    v, s = synth.score_lists(1, 1, N, 8)
    got, st = _select(vs, v, s, 0.8, 0.8, 4096, 65536)
    assert st == 0
    _assert_same(got, oracle.select_topp(v, s, 0.8, 0.8, 4096, 65536))
    with pytest.raises(vs.VSError) as e:
        z = torch.zeros(1, 1, N + 64, device="cuda")
        vs.vs_select_topp(z, z, 0.5, 0.5, 64, 64)
    assert e.value.code == VS_ERR_SHAPE


def test_select_topp_ties_and_extremes(vs):
    N = 1024
    v = np.full((1, 4, N), 1.0 / 16, np.float32)  # equal scores: k = ceil(p N), lowest indices
    s = np.full((1, 4, N), 1.0 / 16, np.float32)
    s[0, 1] = 0.0
    s[0, 1, 300:310] = 6.4  # one pooled block holds all the slash mass
    v[0, 2] = 0.0           # an all-zero list: budget 0 at any p
    v[0, 3, :512] = 0.0     # p = 1 counts the positive entries
    for pv, ps in ((0.25, 0.5), (0.0, 1.0), (1.0, 0.0), (0.07, 0.13)):
        got, st = _select(vs, v, s, pv, ps, N, N)
        assert st == 0
        ref = oracle.select_topp(v, s, pv, ps, N, N)
        _assert_same(got, ref)
    got, _ = _select(vs, v, s, 0.25, 0.5, N, N)
    assert got[2][0, 0] == 256 and np.array_equal(got[0][0, 0, :256], np.arange(256))
    assert got[3][0, 1] == 64 and got[2][0, 2] == 0 and (got[0][0, 2] == -1).all()
    got, _ = _select(vs, v, s, 1.0, 1.0, N, N)
    assert got[2][0, 3] == 512 and np.array_equal(got[0][0, 3, :512], np.arange(512, N))


def test_select_topp_bad_scores(vs):
    N = 512
    v, s = synth.score_lists(1, 3, N, 9)
    v[0, 1, 17] = -1e-3
    s[0, 2, 400] = np.nan
    got, st = _select(vs, v, s, 0.9, 0.9, N, N)
    assert st == VS_ERR_SCORE
    ref = oracle.select_topp(v[:, :1], s[:, :1], 0.9, 0.9, N, N)
    # the bad lists are empty; the good ones are unaffected
    assert got[2][0, 1] == 0 and (got[0][0, 1] == -1).all()
    assert got[3][0, 2] == 0 and (got[1][0, 2] == -1).all()
    np.testing.assert_array_equal(got[0][0, 0], ref[0][0, 0])
    np.testing.assert_array_equal(got[1][0, 0], ref[1][0, 0])


def test_estimate_topp_replay_and_consistency(vs):
    w, x = make_inputs(2, 2048, 4, 2, 64, seed=31, n_out=6, n_slash=5)
    q, k = dev_bf16(x["q"]), dev_bf16(x["k"])
    N, Hq = w.N, w.Hq
    vsc = torch.empty(2, Hq, N, device="cuda")
    ssc = torch.empty(2, Hq, N, device="cuda")
    need = vs.lib().vs_estimate_workspace(ctypes.byref(vs.make_shape(q, k)), 64)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    iv, is_, kv, ks = vs.vs_estimate_topp(q, k, 0.9, 0.8, 1500, 2048, w.scale, v_score=vsc, s_score=ssc, ws=ws)
    torch.cuda.synchronize()
    assert vs.vs_check_status(ws) == 0
    v_gpu, s_gpu = vsc.cpu().numpy(), ssc.cpu().numpy()
    # scores: as in the fixed-budget estimator
    v_ref, s_ref = oracle.estimate(host_f64(x["q"]), host_f64(x["k"]), 64, w.scale)
    assert np.max(np.abs(v_gpu - v_ref)) <= 1e-4 * v_ref.max()
    assert np.max(np.abs(s_gpu - s_ref)) <= 1e-4 * s_ref.max()
    # replay: the oracle's top-p selection on the GPU's own scores
    _assert_same([t.cpu().numpy() for t in (iv, is_, kv, ks)], oracle.select_topp(v_gpu, s_gpu, 0.9, 0.8, 1500, 2048))
    # same scores as the fixed-budget entry point; a fixed budget equal to a
    # head's top-p budget selects the same list
    vsc2 = torch.empty_like(vsc)
    ssc2 = torch.empty_like(ssc)
    kv0 = int(kv[0, 0])
    iv_fixed, _ = vs.vs_estimate(q, k, kv0, 64, w.scale, v_score=vsc2, s_score=ssc2)
    assert torch.equal(vsc, vsc2) and torch.equal(ssc, ssc2)
    assert torch.equal(iv_fixed[0, 0], iv[0, 0, :kv0])
    # the planted outlier columns carry mass: always inside a 90% budget
    ivh = iv.cpu().numpy()
    for b in range(2):
        for h in range(Hq):
            assert set(x["planted_cols"][b][h // 2].tolist()) <= set(ivh[b, h].tolist())


def test_padded_lists_index_and_attention(vs):
    """The oracle's top-p selection (padded lists) through the index builder
    and the attention kernels, against the oracle on the same lists."""
    B, N, Hq, Hkv, d = 1, 1088, 4, 2, 128
    w, x = make_inputs(B, N, Hq, Hkv, d, seed=33, n_out=4, n_slash=3)
    v_ref, s_ref = oracle.estimate(host_f64(x["q"]), host_f64(x["k"]), 64, w.scale)
    iv, is_, kv, ks = oracle.select_topp(v_ref, s_ref, 0.6, 0.5, 200, 512)
    assert (kv < 200).any() and (ks < 512).all()  # padding present
    q, k, vv = dev_bf16(x["q"]), dev_bf16(x["k"]), dev_bf16(x["v"])
    arena = vs.vs_build_block_index(q, k, torch.from_numpy(iv).cuda(), torch.from_numpy(is_).cuda())
    o, lse = vs.vs_attn_fwd(q, k, vv, arena)
    dq, dk, dv = vs.vs_attn_bwd(q, k, vv, o, lse, dev_bf16(x["dout"]), arena, 200)
    torch.cuda.synchronize()
    assert vs.vs_check_status(arena) == 0
    A = Arena(arena)
    p = oracle.Problem(host_f64(x["q"]), host_f64(x["k"]), host_f64(x["v"]), iv, is_, w.scale,
                       dout=host_f64(x["dout"]))
    for h in range(Hq):
        M = oracle.mask_dense(p, 0, h).astype(np.int32)
        np.testing.assert_array_equal(A.coverage_query_major(h), M)
        np.testing.assert_array_equal(A.coverage_key_major(h), M)
    ref = oracle.attention(p)
    for name, got in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert rel_l2(host_f64(got), ref[name]) <= 1e-2, name
    fin = np.isfinite(ref["lse"])
    lse_h = lse.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(np.isfinite(lse_h), fin)
    assert np.max(np.abs(lse_h[fin] - ref["lse"][fin]), initial=0.0) <= 1e-3


def test_index_padding_rules(vs):
    N = 256
    q = torch.zeros(1, N, 2, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, N, 1, 64, dtype=torch.bfloat16, device="cuda")
    # all-padding lists: the empty mask
    iv = torch.full((1, 2, 5), -1, dtype=torch.int32, device="cuda")
    is_ = torch.full((1, 2, 3), -1, dtype=torch.int32, device="cuda")
    arena = vs.vs_build_block_index(q, k, iv, is_)
    torch.cuda.synchronize()
    assert vs.vs_check_status(arena) == 0
    A = Arena(arena)
    assert (A.counts == 0).all() and (A.vcount == 0).all() and (A.ecount == 0).all()
    o, lse = vs.vs_attn_fwd(q, k, torch.zeros_like(k), arena)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    # an entry after a -1 is rejected; so is any other negative value
    for bad in ([3, -1, 7], [3, -2, -1]):
        arena = vs.vs_build_block_index(q, k, torch.tensor([[bad, bad]], dtype=torch.int32, device="cuda"), is_)
        torch.cuda.synchronize()
        assert vs.vs_check_status(arena) == VS_ERR_INDEX


def test_vsattention_topp_mode(vs):
    """The layer object in top-p mode: its budgets and lists replay through
    the oracle's selection on its own scores, and a forward / backward on
    the oracle's selection (passed in) matches the oracle."""
    w, x = make_inputs(1, 2048, 4, 2, 128, seed=35, n_out=5, n_slash=4)
    layer = vs.VSAttention(1, 2048, 4, 2, 128, 600, 1024, pv=0.85, ps=0.7)
    q, k, v = dev_bf16(x["q"]), dev_bf16(x["k"]), dev_bf16(x["v"])
    layer.forward(q, k, v)
    layer.backward(dev_bf16(x["dout"]))
    torch.cuda.synchronize()
    layer.check()
    got = [layer.v_idx.cpu().numpy(), layer.s_idx.cpu().numpy(), layer.budgets[0].cpu().numpy(),
           layer.budgets[1].cpu().numpy()]
    _assert_same(got, oracle.select_topp(layer.v_score.cpu().numpy(), layer.s_score.cpu().numpy(), 0.85, 0.7, 600,
                                         1024))
    v_ref, s_ref = oracle.estimate(host_f64(x["q"]), host_f64(x["k"]), 64, w.scale)
    iv, is_, _, _ = oracle.select_topp(v_ref, s_ref, 0.85, 0.7, 600, 1024)
    o, lse = layer.forward(q, k, v, selection=(torch.from_numpy(iv).cuda(), torch.from_numpy(is_).cuda()))
    dq, dk, dv = layer.backward(dev_bf16(x["dout"]))
    torch.cuda.synchronize()
    layer.check()
    ref = oracle.attention(oracle.Problem(host_f64(x["q"]), host_f64(x["k"]), host_f64(x["v"]), iv, is_, w.scale,
                                          dout=host_f64(x["dout"])))
    for name, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert rel_l2(host_f64(t), ref[name]) <= 1e-2, name
