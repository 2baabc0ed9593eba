"""GQA head packing (VS_INDEX_PACK_GQA) on a per-KV-group selection: the
query-major tiles hold 128 / g tokens of the g query heads of a KV group.
The mask is unchanged, so O, LSE, dQ, dK, dV must match the fp64 oracle on
the same (group-shared) selection, and the unpacked path; the index refuses
lists that differ inside a group."""
import math

import numpy as np
import pytest
import torch

import oracle
from vs_testutil import dev_bf16, host_f64, make_inputs, rel_l2

pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module")
def vs():
    import dynamic_vertical_slash_gb300 as m

    return m


def _group_selection(B, Hq, Hkv, N, kv, ks, seed):
    """One random selection per KV group, repeated for the group's heads."""
    rng = np.random.default_rng(seed)
    g = Hq // Hkv
    iv = np.zeros((B, Hq, kv), np.int32)
    is_ = np.zeros((B, Hq, ks), np.int32)
    for b in range(B):
        for hk in range(Hkv):
            a = np.sort(rng.choice(N, kv, replace=False))
            c = np.sort(rng.choice(N, ks, replace=False))
            iv[b, hk * g:(hk + 1) * g] = a
            is_[b, hk * g:(hk + 1) * g] = c
    return iv, is_


def _run(vs, x, iv, is_, d, pack):
    q, k, v, do = (dev_bf16(x[n]) for n in ("q", "k", "v", "dout"))
    ivd, isd = torch.from_numpy(iv).cuda(), torch.from_numpy(is_).cuda()
    arena = vs.vs_build_block_index(q, k, ivd, isd, pack_gqa=pack)
    o, lse = vs.vs_attn_fwd(q, k, v, arena)
    dq, dk, dv = vs.vs_attn_bwd(q, k, v, o, lse, do, arena, iv.shape[-1])
    torch.cuda.synchronize()
    assert vs.vs_check_status(arena) == 0
    return {"o": host_f64(o), "lse": lse.cpu().numpy().astype(np.float64), "dq": host_f64(dq), "dk": host_f64(dk),
            "dv": host_f64(dv), "counts": vs.vs_index_counts(arena)}


@pytest.mark.parametrize("B,N,Hq,Hkv,d,kv,ks", [
    (1, 1088, 8, 1, 64, 24, 40),     # g = 8 (16-token strips), ragged last 128-row tile
    (2, 1024, 16, 2, 128, 30, 64),   # the Qwen2.5-3B grouping, two batches
    (1, 1024, 4, 2, 64, 16, 48),     # g = 2 (64-token strips)
    (1, 1024, 8, 2, 128, 1, 1),      # g = 4, budgets of one
])
def test_packed_matches_oracle_and_unpacked(vs, B, N, Hq, Hkv, d, kv, ks):
    w, x = make_inputs(B, N, Hq, Hkv, d, seed=71 + N + Hq, n_out=3, n_slash=2)
    iv, is_ = _group_selection(B, Hq, Hkv, N, kv, ks, 72 + Hq)
    got = _run(vs, x, iv, is_, d, True)
    ref = oracle.attention(oracle.Problem(host_f64(x["q"]), host_f64(x["k"]), host_f64(x["v"]), iv, is_,
                                          1 / math.sqrt(d), dout=host_f64(x["dout"])))
    for name in ("o", "dq", "dk", "dv"):
        assert rel_l2(got[name], ref[name]) <= TOL, name
    fin = np.isfinite(ref["lse"])
    np.testing.assert_array_equal(np.isfinite(got["lse"]), fin)
    assert np.max(np.abs(got["lse"][fin] - ref["lse"][fin]), initial=0.0) <= 1e-3
    # the same mask through one-head-per-tile kernels
    unp = _run(vs, x, iv, is_, d, False)
    for name in ("o", "dq", "dk", "dv"):
        assert rel_l2(got[name], unp[name]) <= TOL, name
    # query-major work: reported at each group's first head; the key-major
    # (dK / dV) cover is the same in both
    g = Hq // Hkv
    cp, cu = got["counts"].reshape(B, Hq, 4), unp["counts"].reshape(B, Hq, 4)
    assert np.all(cp[:, [h for h in range(Hq) if h % g], :2] == 0)
    np.testing.assert_array_equal(cp[..., 2:], cu[..., 2:])
    assert cp[..., 0].sum() <= cu[..., 0].sum()


def test_packed_index_refuses_lists_that_differ_in_a_group(vs):
    B, N, Hq, Hkv, d = 1, 512, 4, 1, 64
    w, x = make_inputs(B, N, Hq, Hkv, d, seed=81)
    iv, is_ = _group_selection(B, Hq, Hkv, N, 8, 8, 82)
    # head 3's slash list: one offset swapped for one it does not hold (still
    # sorted and unique, so only the group rule can reject it)
    free = np.setdiff1d(np.arange(N), is_[0, 3])[0]
    is_[0, 3, 0] = free
    is_[0, 3] = np.sort(is_[0, 3])
    q, k = dev_bf16(x["q"]), dev_bf16(x["k"])
    arena = vs.vs_build_block_index(q, k, torch.from_numpy(iv).cuda(), torch.from_numpy(is_).cuda(), pack_gqa=True)
    torch.cuda.synchronize()
    assert vs.vs_check_status(arena) == 4  # VS_ERR_INDEX


def test_layer_with_packed_heads(vs):
    # VSAttention(shared=True, packed=True): the estimator's group selection
    # through packed tiles equals the same selection unpacked
    B, N, Hq, Hkv, d = 1, 2048, 8, 1, 64
    w, x = make_inputs(B, N, Hq, Hkv, d, seed=91, n_out=6, n_slash=3)
    q, k, v, do = (dev_bf16(x[n]) for n in ("q", "k", "v", "dout"))
    outs = []
    for packed in (False, True):
        att = vs.VSAttention(B, N, Hq, Hkv, d, 32, 64, shared=True, packed=packed)
        o, lse = att.forward(q, k, v)
        dq, dk, dv = att.backward(do)
        torch.cuda.synchronize()
        att.check()
        outs.append([host_f64(t) for t in (o, dq, dk, dv)] + [att.v_idx.cpu().numpy(), att.s_idx.cpu().numpy()])
    assert np.array_equal(outs[0][4], outs[1][4]) and np.array_equal(outs[0][5], outs[1][5])
    for a, b in zip(outs[0][:4], outs[1][:4]):
        assert rel_l2(b, a) <= TOL
    iv, is_ = outs[1][4], outs[1][5]
    ref = oracle.attention(oracle.Problem(host_f64(x["q"]), host_f64(x["k"]), host_f64(x["v"]), iv, is_,
                                          1 / math.sqrt(d), dout=host_f64(x["dout"])))
    for got, name in zip(outs[1][:4], ("o", "dq", "dk", "dv")):
        assert rel_l2(got, ref[name]) <= TOL, name
