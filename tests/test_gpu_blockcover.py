"""Block-cover reading of the slashes on the GPU (MTraining section 4.1 (ii):
slashes taken at the granularity of 64 x 64 blocks) against the oracle's
block mask, through the C ABI: exact index coverage, forward and backward
parity unstriped and on striped ring steps, and the exact-mask path left as
it was."""
import math

import numpy as np
import pytest
import torch

import oracle
from vs_testutil import Arena, dev_bf16, host_f64, make_inputs, random_selection, rel_l2

pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module")
def vs():
    import dynamic_vertical_slash_gb300 as m

    m.lib()
    return m


def _problem(x, iv, is_, d, **kw):
    return oracle.Problem(host_f64(x["q"]), host_f64(x["k"]), host_f64(x["v"]), iv, is_, 1 / math.sqrt(d),
                          dout=host_f64(x["dout"]), block=True, **kw)


def _compare(got, ref):
    for key in ("o", "dq", "dk", "dv"):
        assert rel_l2(host_f64(got[key]), ref[key]) <= TOL, key
    lse = got["lse"].cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref["lse"])
    np.testing.assert_array_equal(np.isfinite(lse), fin)
    assert np.max(np.abs(lse[fin] - ref["lse"][fin]), initial=0.0) <= 1e-3


# active block diagonals D at given spacings: an offset 64 D activates only
# diagonal D, and the dilated offset intervals of diagonals k apart overlap
# (k <= 3), are just separated (k = 4: the previous cover interval overhangs
# the next one) or are entered at their own start (k >= 5)
@pytest.mark.parametrize("steps", [(1,), (3,), (4,), (5,), (6,), (1, 4, 2, 5, 3, 6)])
def test_block_index_cover_diagonal_spacings(vs, steps):
    N, Hq, Hkv, d, kv = 2560, 2, 1, 64, 4
    diags, D, i = [], 1, 0
    while 64 * D < N:
        diags.append(D)
        D += steps[i % len(steps)]
        i += 1
    offs = [64 * D for D in diags]
    ks = len(offs)
    is_ = np.full((1, Hq, ks), -1, np.int32)
    is_[0, 0] = offs
    is_[0, 1, :ks - 1] = offs[1:]  # the other head: without the first diagonal
    rng = np.random.default_rng(len(steps))
    iv = np.sort(rng.choice(N, size=(1, Hq, kv), replace=False), axis=-1).astype(np.int32)
    q = torch.zeros(1, N, Hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, N, Hkv, d, dtype=torch.bfloat16, device="cuda")
    arena = vs.vs_build_block_index(q, k, torch.from_numpy(iv).cuda(), torch.from_numpy(is_).cuda(),
                                    block_cover=True)
    torch.cuda.synchronize()
    assert vs.vs_check_status(arena) == 0
    A = Arena(arena)
    p = oracle.Problem(np.zeros((1, N, Hq, d)), np.zeros((1, N, Hkv, d)), np.zeros((1, N, Hkv, d)), iv, is_, 0.1,
                       block=True)
    for h in range(Hq):
        M = oracle.mask_dense(p, 0, h).astype(np.int32)
        np.testing.assert_array_equal(A.coverage_query_major(h), M)
        np.testing.assert_array_equal(A.coverage_key_major(h), M)


@pytest.mark.parametrize("N,kv,ks,seed", [(1024, 32, 32, 1), (1088, 40, 50, 2), (640, 3, 200, 3), (256, 4, 1, 4)])
def test_block_index_covers_block_mask_exactly_once(vs, N, kv, ks, seed):
    Hq, Hkv, d = 2, 1, 64
    iv, is_ = random_selection(1, Hq, N, kv, ks, seed)
    q = torch.zeros(1, N, Hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, N, Hkv, d, dtype=torch.bfloat16, device="cuda")
    arena = vs.vs_build_block_index(q, k, torch.from_numpy(iv).cuda(), torch.from_numpy(is_).cuda(),
                                    block_cover=True)
    torch.cuda.synchronize()
    assert vs.vs_check_status(arena) == 0
    A = Arena(arena)
    assert A.block_cover == 1
    p = oracle.Problem(np.zeros((1, N, Hq, d)), np.zeros((1, N, Hkv, d)), np.zeros((1, N, Hkv, d)), iv, is_, 0.1,
                       block=True)
    for h in range(Hq):
        M = oracle.mask_dense(p, 0, h).astype(np.int32)
        np.testing.assert_array_equal(A.coverage_query_major(h), M)
        np.testing.assert_array_equal(A.coverage_key_major(h), M)


@pytest.mark.parametrize("B,N,Hq,Hkv,d,kv,ks,seed", [
    (1, 1088, 4, 2, 128, 40, 50, 5),   # ragged query tile, GQA
    (2, 640, 8, 1, 64, 13, 9, 6),      # g = 8, few slashes: whole blocks dominate
    (1, 384, 2, 2, 128, 1, 1, 7),
])
def test_block_attention_parity(vs, B, N, Hq, Hkv, d, kv, ks, seed):
    w, x = make_inputs(B, N, Hq, Hkv, d, seed, n_out=4, n_slash=3)
    iv, is_ = random_selection(B, Hq, N, kv, ks, seed + 100)
    q, k, v = dev_bf16(x["q"]), dev_bf16(x["k"]), dev_bf16(x["v"])
    arena = vs.vs_build_block_index(q, k, torch.from_numpy(iv).cuda(), torch.from_numpy(is_).cuda(),
                                    block_cover=True)
    o, lse = vs.vs_attn_fwd(q, k, v, arena)
    dq, dk, dv = vs.vs_attn_bwd(q, k, v, o, lse, dev_bf16(x["dout"]), arena, kv)
    torch.cuda.synchronize()
    assert vs.vs_check_status(arena) == 0
    ref = oracle.attention(_problem(x, iv, is_, d))
    _compare({"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}, ref)
    # the block mask holds the exact one: more entries, different result
    exact = oracle.attention(oracle.Problem(host_f64(x["q"]), host_f64(x["k"]), host_f64(x["v"]), iv, is_,
                                            1 / math.sqrt(d)))
    assert rel_l2(ref["o"], exact["o"]) > 1e-3


def test_block_striped_ring_steps_match_global(vs):
    """Worker 0 of W: W ring steps with merge and dQ accumulation in block
    mode equal the global block-mask computation on worker 0's rows."""
    B, N, Hq, Hkv, d, W = 1, 2048, 2, 1, 64, 4
    w, x = make_inputs(B, N, Hq, Hkv, d, seed=22, n_out=4, n_slash=3)
    iv, is_ = random_selection(B, Hq, N, 24, 20, 23)
    ref = oracle.attention(_problem(x, iv, is_, d))
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
        arena = vs.vs_build_block_index(qs, ks_[src], ivd, isd, vs.make_stripe(W, 0, src, N), block_cover=True)
        arenas.append((src, arena))
        vs.vs_attn_fwd(qs, ks_[src], vs_[src], arena, o=o, lse=lse, o_acc=o_acc)
    pos = oracle.stripe_positions(N, W, 64, 0)
    torch.cuda.synchronize()
    assert rel_l2(host_f64(o)[0], ref["o"][0, pos]) <= TOL
    fin = np.isfinite(ref["lse"][0][:, pos])
    assert np.max(np.abs(lse.cpu().numpy()[0][fin] - ref["lse"][0][:, pos][fin])) <= 1e-3
    dq_acc = torch.zeros(B, Nl, Hq, d, device="cuda")
    dq = torch.empty_like(qs)
    for src, arena in arenas:
        vs.vs_attn_bwd(qs, ks_[src], vs_[src], o, lse, dos, arena, 24, dq=dq, dq_acc=dq_acc)
    torch.cuda.synchronize()
    assert rel_l2(host_f64(dq)[0], ref["dq"][0, pos]) <= TOL
    for src, arena in arenas:
        assert vs.vs_check_status(arena) == 0


def test_layer_block_cover_option(vs):
    w, x = make_inputs(1, 1024, 4, 2, 64, seed=41, n_out=4, n_slash=3)
    q, k, v = dev_bf16(x["q"]), dev_bf16(x["k"]), dev_bf16(x["v"])
    iv, is_ = random_selection(1, 4, 1024, 20, 30, 42)
    layer = vs.VSAttention(1, 1024, 4, 2, 64, 20, 30, block_cover=True)
    o, lse = layer.forward(q, k, v, selection=(torch.from_numpy(iv).cuda(), torch.from_numpy(is_).cuda()))
    dq, dk, dv = layer.backward(dev_bf16(x["dout"]))
    torch.cuda.synchronize()
    layer.check()
    _compare({"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}, oracle.attention(_problem(x, iv, is_, 64)))
