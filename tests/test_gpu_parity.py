"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Tolerances: O, dQ, dK, dV relative L2 <= 1e-2 (bf16 inputs, fp32
accumulation); LSE absolute <= 1e-3; estimator scores within 1e-4 of the
largest score; selected indices bit-exact under the replay rule (the oracle's
top-k applied to the GPU's own fp32 scores) and equal to the oracle's own
selection on planted inputs; index coverage exact (every mask entry computed
exactly once).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from vs_testutil import Arena, dev_bf16, host_f64, make_inputs, random_selection, rel_l2

pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module")
def vs():
    import dynamic_vertical_slash_gb300 as m

    m.lib()
    return m


def _run_attention(vs, x, iv, is_, kv, stripe=None, bwd=True):
    q, k, v = dev_bf16(x["q"]), dev_bf16(x["k"]), dev_bf16(x["v"])
    ivd = torch.from_numpy(iv).cuda()
    isd = torch.from_numpy(is_).cuda()
    arena = vs.vs_build_block_index(q, k, ivd, isd, stripe)
    o, lse = vs.vs_attn_fwd(q, k, v, arena)
    out = {"o": o, "lse": lse, "arena": arena}
    if bwd:
        do = dev_bf16(x["dout"])
        dq, dk, dv = vs.vs_attn_bwd(q, k, v, o, lse, do, arena, kv)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert vs.vs_check_status(arena) == 0
    return out


def _oracle_problem(x, iv, is_, d):
    return oracle.Problem(host_f64(x["q"]), host_f64(x["k"]), host_f64(x["v"]), iv, is_, 1 / math.sqrt(d),
                          dout=host_f64(x["dout"]))


def _compare(out, ref, what=("o", "dq", "dk", "dv")):
    for key in what:
        err = rel_l2(host_f64(out[key]), ref[key])
        assert err <= TOL, (key, err)
    lse = out["lse"].cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref["lse"])
    np.testing.assert_array_equal(np.isfinite(lse), fin)
    assert np.max(np.abs(lse[fin] - ref["lse"][fin]), initial=0.0) <= 1e-3


# ---------------------------------------------------------------- estimator
def test_estimate_tiny_workload_parity(vs):
    w = synth.workloads()["tiny-1k"]
    x = synth.make_batch(w)
    q, k = dev_bf16(x["q"]), dev_bf16(x["k"])
    B, N, Hq = w.B, w.N, w.Hq
    vsc = torch.empty(B, Hq, N, device="cuda")
    ssc = torch.empty(B, Hq, N, device="cuda")
    iv, is_ = vs.vs_estimate(q, k, w.kv, w.ks, w.scale, 64, v_score=vsc, s_score=ssc)
    torch.cuda.synchronize()
    v_ref, s_ref = oracle.estimate(host_f64(x["q"]), host_f64(x["k"]), 64, w.scale)
    v_gpu, s_gpu = vsc.cpu().numpy(), ssc.cpu().numpy()
    assert np.max(np.abs(v_gpu - v_ref)) <= 1e-4 * v_ref.max()
    assert np.max(np.abs(s_gpu - s_ref)) <= 1e-4 * s_ref.max()
    ivh, ish = iv.cpu().numpy(), is_.cpu().numpy()
    for b in range(B):
        for h in range(Hq):
            # replay: the oracle's selection rule on the GPU's own scores is bit-exact
            np.testing.assert_array_equal(ivh[b, h], oracle.topk(v_gpu[b, h], w.kv))
            np.testing.assert_array_equal(ish[b, h], oracle.topk(s_gpu[b, h], w.ks))
            # the planted outlier columns are always selected
            assert set(x["planted_cols"][b][0].tolist()) <= set(ivh[b, h].tolist())
    # budget equal to the planted count: exactly the planted columns
    iv8, _ = vs.vs_estimate(q, k, 8, 8, w.scale)
    for h in range(Hq):
        np.testing.assert_array_equal(iv8.cpu().numpy()[0, h], x["planted_cols"][0][0])


def test_estimate_selection_matches_oracle_on_planted_slashes(vs):
    w, x = make_inputs(1, 2048, 4, 2, 64, seed=21, n_out=6, n_slash=5)
    q, k = dev_bf16(x["q"]), dev_bf16(x["k"])
    v_ref, s_ref = oracle.estimate(host_f64(x["q"]), host_f64(x["k"]), 64, w.scale)
    iv_ref, is_ref = oracle.select(v_ref, s_ref, 6, 5)
    iv, is_ = vs.vs_estimate(q, k, 6, 5, w.scale)
    np.testing.assert_array_equal(iv.cpu().numpy(), iv_ref)
    np.testing.assert_array_equal(is_.cpu().numpy(), is_ref)


def test_topk_ties_lowest_index(vs):
    # equal scores everywhere: the lowest indices win (K = 0 gives uniform rows
    # whose column sums tie in runs)
    N = 512
    q = torch.randn(1, N, 1, 64, device="cuda").to(torch.bfloat16)
    k = torch.zeros(1, N, 1, 64, device="cuda", dtype=torch.bfloat16)
    vsc = torch.empty(1, 1, N, device="cuda")
    ssc = torch.empty(1, 1, N, device="cuda")
    iv, is_ = vs.vs_estimate(q, k, 100, 77, 0.125, v_score=vsc, s_score=ssc)
    np.testing.assert_array_equal(iv.cpu().numpy()[0, 0], oracle.topk(vsc.cpu().numpy()[0, 0], 100))
    np.testing.assert_array_equal(is_.cpu().numpy()[0, 0], oracle.topk(ssc.cpu().numpy()[0, 0], 77))


# -------------------------------------------------------------------- index
@pytest.mark.parametrize("N,kv,ks,seed", [(1024, 32, 32, 1), (1088, 40, 50, 2), (640, 3, 200, 3), (256, 256, 1, 4)])
def test_index_covers_mask_exactly_once(vs, N, kv, ks, seed):
    Hq, Hkv, d = 2, 1, 64
    iv, is_ = random_selection(1, Hq, N, kv, ks, seed)
    q = torch.zeros(1, N, Hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, N, Hkv, d, dtype=torch.bfloat16, device="cuda")
    arena = vs.vs_build_block_index(q, k, torch.from_numpy(iv).cuda(), torch.from_numpy(is_).cuda())
    A = Arena(arena)
    p = oracle.Problem(np.zeros((1, N, Hq, d)), np.zeros((1, N, Hkv, d)), np.zeros((1, N, Hkv, d)), iv, is_, 0.1)
    for h in range(Hq):
        M = oracle.mask_dense(p, 0, h).astype(np.int32)
        np.testing.assert_array_equal(A.coverage_query_major(h), M)
        np.testing.assert_array_equal(A.coverage_key_major(h), M)


# slash offsets whose gaps sit at the boundaries of the cover's segments: the
# dilated intervals [o, o + 127] touch (gap 128), just separate (129, 130),
# leave the previous cover interval overhanging the next segment (gap 190:
# 63 past the segment's end) or not (191: exactly 64; 192)
@pytest.mark.parametrize("gaps", [(65,), (128,), (129,), (130,), (190,), (191,), (192,), (1, 190, 63, 191, 300),
                                  (127, 128, 129, 190, 191, 192, 64, 65, 2)])
def test_index_cover_segment_gaps(vs, gaps):
    N, Hq, Hkv, d, kv = 1536, 2, 1, 64, 8
    offs, o, i = [], 3, 0
    while o < N:
        offs.append(o)
        o += gaps[i % len(gaps)]
        i += 1
    ks = len(offs)
    is_ = np.full((1, Hq, ks), -1, np.int32)
    is_[0, 0] = offs
    is_[0, 1, :ks // 2] = offs[::2][:ks // 2]  # the other head: every second offset
    rng = np.random.default_rng(len(gaps))
    iv = np.sort(rng.choice(N, size=(1, Hq, kv), replace=False), axis=-1).astype(np.int32)
    q = torch.zeros(1, N, Hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, N, Hkv, d, dtype=torch.bfloat16, device="cuda")
    arena = vs.vs_build_block_index(q, k, torch.from_numpy(iv).cuda(), torch.from_numpy(is_).cuda())
    torch.cuda.synchronize()
    assert vs.vs_check_status(arena) == 0
    A = Arena(arena)
    p = oracle.Problem(np.zeros((1, N, Hq, d)), np.zeros((1, N, Hkv, d)), np.zeros((1, N, Hkv, d)), iv, is_, 0.1)
    for h in range(Hq):
        M = oracle.mask_dense(p, 0, h).astype(np.int32)
        np.testing.assert_array_equal(A.coverage_query_major(h), M)
        np.testing.assert_array_equal(A.coverage_key_major(h), M)


def test_index_rejects_bad_lists(vs):
    N = 256
    q = torch.zeros(1, N, 1, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, N, 1, 64, dtype=torch.bfloat16, device="cuda")
    iv = torch.tensor([[[5, 3, 9]]], dtype=torch.int32, device="cuda")  # unsorted
    is_ = torch.tensor([[[0, 1]]], dtype=torch.int32, device="cuda")
    arena = vs.vs_build_block_index(q, k, iv, is_)
    # attention on a rejected arena does nothing and reports the error
    v = torch.zeros_like(k)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    vs.vs_attn_fwd(q, k, v, arena, ws=ws)
    torch.cuda.synchronize()
    assert vs.vs_check_status(arena) == 4
    assert vs.vs_check_status(ws) == 4
    iv2 = torch.tensor([[[5, 300, 9000]]], dtype=torch.int32, device="cuda")  # out of range
    arena = vs.vs_build_block_index(q, k, iv2, is_)
    torch.cuda.synchronize()
    assert vs.vs_check_status(arena) == 4


# ---------------------------------------------------------------- attention
def test_tiny_workload_end_to_end(vs):
    """The 1K workload: GPU selection equals the oracle's; attention on it
    matches the oracle within tolerance."""
    w = synth.workloads()["tiny-1k"]
    x = synth.make_batch(w)
    v_ref, s_ref = oracle.estimate(host_f64(x["q"]), host_f64(x["k"]), 64, w.scale)
    iv, is_ = oracle.select(v_ref, s_ref, w.kv, w.ks)
    q, k = dev_bf16(x["q"]), dev_bf16(x["k"])
    ivg, isg = vs.vs_estimate(q, k, w.kv, w.ks, w.scale)
    # fp32 scores on the GPU vs fp64 in the oracle: selections may differ only
    # between indices whose oracle scores lie within the fp32 error of the
    # k-th score
    for sel_g, sel_o, sc, kk in ((ivg, iv, v_ref, w.kv), (isg, is_, s_ref, w.ks)):
        sel_g = sel_g.cpu().numpy()
        for h in range(w.Hq):
            diff = np.setxor1d(sel_g[0, h], sel_o[0, h])
            kth = np.sort(sc[0, h])[::-1][kk - 1]
            assert np.all(np.abs(sc[0, h][diff] - kth) <= 1e-5 * sc[0, h].max()), diff
    out = _run_attention(vs, x, iv, is_, w.kv)
    _compare(out, oracle.attention(_oracle_problem(x, iv, is_, w.d)))


@pytest.mark.parametrize("B,N,Hq,Hkv,d,kv,ks,seed", [
    (2, 1088, 4, 2, 128, 40, 50, 5),    # ragged query tile, GQA, d=128, batch 2
    (1, 640, 8, 1, 64, 13, 90, 6),      # g = 8
    (1, 384, 2, 2, 128, 1, 1, 7),       # tiny budgets: many empty rows
])
def test_attention_parity_random_selection(vs, B, N, Hq, Hkv, d, kv, ks, seed):
    w, x = make_inputs(B, N, Hq, Hkv, d, seed, n_out=4, n_slash=3)
    iv, is_ = random_selection(B, Hq, N, kv, ks, seed + 100)
    out = _run_attention(vs, x, iv, is_, kv)
    _compare(out, oracle.attention(_oracle_problem(x, iv, is_, d)))


def test_dense_fallback_equals_dense_attention(vs):
    """ks = N selects every offset: the mask is the full causal mask and the
    result equals dense causal attention (library SDPA as a cross-check)."""
    B, N, Hq, Hkv, d = 1, 512, 4, 2, 128
    w, x = make_inputs(B, N, Hq, Hkv, d, seed=8, n_out=3)
    iv, _ = random_selection(B, Hq, N, 16, 1, 9)
    is_ = np.tile(np.arange(N, dtype=np.int32), (B, Hq, 1))
    out = _run_attention(vs, x, iv, is_, 16)
    ref = oracle.attention(_oracle_problem(x, iv, is_, d))
    _compare(out, ref)
    qf, kf, vf = (torch.from_numpy(host_f64(x[n])).transpose(1, 2) for n in ("q", "k", "v"))
    sdpa = torch.nn.functional.scaled_dot_product_attention(qf, kf.repeat_interleave(2, 1), vf.repeat_interleave(2, 1),
                                                            is_causal=True)
    assert rel_l2(host_f64(out["o"]), sdpa.transpose(1, 2).numpy()) <= TOL


def test_single_and_empty_rows(vs):
    N, d = 256, 64
    w, x = make_inputs(1, N, 1, 1, d, seed=10)
    iv = np.array([[[200]]], np.int32)
    is_ = np.array([[[7]]], np.int32)
    out = _run_attention(vs, x, iv, is_, 1)
    ref = oracle.attention(_oracle_problem(x, iv, is_, d))
    _compare(out, ref)
    o = host_f64(out["o"])
    assert np.all(o[0, :7] == 0)  # rows 0..6 see nothing
    np.testing.assert_allclose(o[0, 7, 0], host_f64(x["v"])[0, 0, 0], rtol=0, atol=0)  # one entry: exact copy of v


# ------------------------------------------------------------------ striped
def test_striped_permute_matches_oracle(vs):
    B, N, H, d, W = 2, 2048, 3, 64, 4
    x = torch.randn(B, N, H, d, device="cuda").to(torch.bfloat16)
    y = vs.striped_permute(x, W)
    ref = oracle.striped_permute(x.view(torch.int16).cpu().numpy(), W, 64)
    np.testing.assert_array_equal(y.view(torch.int16).cpu().numpy(), ref)
    back = vs.striped_permute(y, W, inverse=True)
    assert torch.equal(back.view(torch.int16), x.view(torch.int16))
    one = vs.striped_permute(x, W, only_rank=2)
    assert torch.equal(one.view(torch.int16), y[2].view(torch.int16))


def test_striped_ring_steps_match_global(vs):
    """Worker 0 of W runs W ring steps (src = -s mod W) with merge mode; the
    merged output equals the global computation on worker 0's rows, and the
    accumulated dQ equals the global dQ on those rows."""
    B, N, Hq, Hkv, d, W = 1, 2048, 2, 1, 64, 4
    w, x = make_inputs(B, N, Hq, Hkv, d, seed=12, n_out=4, n_slash=3)
    iv, is_ = random_selection(B, Hq, N, 24, 40, 13)
    ref = oracle.attention(_oracle_problem(x, iv, is_, d))
    q, k, v, do = (dev_bf16(x[n]) for n in ("q", "k", "v", "dout"))
    qs = vs.striped_permute(q, W, only_rank=0)
    dos = vs.striped_permute(do, W, only_rank=0)
    ks_, vs_ = vs.striped_permute(k, W), vs.striped_permute(v, W)
    ivd, isd = torch.from_numpy(iv).cuda(), torch.from_numpy(is_).cuda()
    Nl = N // W
    o = torch.empty_like(qs)
    lse = torch.full((B, Hq, Nl), -math.inf, device="cuda")
    o_acc = torch.zeros(B, Nl, Hq, d, device="cuda")
    arenas = []
    for s_ in range(W):
        src = (0 - s_) % W
        st = vs.make_stripe(W, 0, src, N)
        arena = vs.vs_build_block_index(qs, ks_[src], ivd, isd, st)
        arenas.append((src, arena))
        vs.vs_attn_fwd(qs, ks_[src], vs_[src], arena, o=o, lse=lse, o_acc=o_acc)
    pos = oracle.stripe_positions(N, W, 64, 0)
    torch.cuda.synchronize()
    assert rel_l2(host_f64(o)[0], ref["o"][0, pos]) <= TOL
    fin = np.isfinite(ref["lse"][0][:, pos])
    assert np.max(np.abs(lse.cpu().numpy()[0][fin] - ref["lse"][0][:, pos][fin])) <= 1e-3
    dq_acc = torch.zeros(B, Nl, Hq, d, device="cuda")
    dq = torch.empty_like(qs)
    dks = {}
    for src, arena in arenas:
        _, dk, dv = vs.vs_attn_bwd(qs, ks_[src], vs_[src], o, lse, dos, arena, 24, dq=dq, dq_acc=dq_acc)
        dks[src] = (dk.clone(), dv.clone())
    torch.cuda.synchronize()
    assert rel_l2(host_f64(dq)[0], ref["dq"][0, pos]) <= TOL
    # dK / dV of shard src from worker 0's queries: the global-normalised
    # contribution of those rows.  The oracle gets worker 0's rows against
    # every key (so its LSE and D are the global ones) and reports the keys
    # of shard src.
    p = oracle.Problem(host_f64(x["q"])[:, pos], host_f64(x["k"]), host_f64(x["v"]), iv, is_, 1 / math.sqrt(d),
                       dout=host_f64(x["dout"])[:, pos], qpos=pos, n_global=N)
    for src in (0, 1, 3):
        kpos = oracle.stripe_positions(N, W, 64, src)
        keys = np.array([(0, 0, m) for m in kpos], np.int32)
        dk_ref, dv_ref = oracle.keys(p, keys)
        assert rel_l2(host_f64(dks[src][0])[0, :, 0], dk_ref) <= TOL, src
        assert rel_l2(host_f64(dks[src][1])[0, :, 0], dv_ref) <= TOL, src
