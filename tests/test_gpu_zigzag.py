"""ZigZag ring on one GPU (MTraining section 2, Figure 1: 2W chunks, worker r
holds chunks r and 2W - 1 - r).  The ZigZag permute against the oracle's
layout, bit for bit; and one worker's ring steps (chunk pairs as windowed
problems on global positions, forward merge, dQ and dK / dV accumulation)
against the fp64 oracle's global computation on the worker's rows."""
import math

import numpy as np
import pytest
import torch

import oracle
from vs_testutil import dev_bf16, host_f64, make_inputs, random_selection, rel_l2

pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module")
def vs():
    import dynamic_vertical_slash_gb300 as m

    return m


def test_ring_permute_zigzag_bit_exact(vs):
    B, N, H, d, W = 2, 2048, 3, 64, 4
    g = torch.Generator().manual_seed(3)
    x = torch.randn(B, N, H, d, generator=g).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy()
    want = oracle.ring_permute(bits, W, "zigzag")
    y = vs.ring_permute(x.cuda(), W, "zigzag")
    assert np.array_equal(y.cpu().view(torch.int16).numpy(), want)
    one = vs.ring_permute(x.cuda(), W, "zigzag", only_rank=2)
    assert np.array_equal(one.cpu().view(torch.int16).numpy(), want[2])
    back = vs.ring_permute(y, W, "zigzag", inverse=True)
    assert torch.equal(back.cpu().view(torch.int16), x.view(torch.int16))
    # the striped layout through the same entry point equals striped_permute
    assert torch.equal(vs.ring_permute(x.cuda(), W, "striped").cpu(), vs.striped_permute(x.cuda(), W).cpu())


@pytest.mark.parametrize("B,rank,d,Hq", [(1, 0, 64, 2), (1, 1, 64, 2), (1, 3, 128, 8), (2, 2, 64, 2)])
def test_zigzag_worker_matches_global(vs, B, rank, d, Hq):
    N, Hkv, W = 2048, 1, 4
    w, x = make_inputs(B, N, Hq, Hkv, d, seed=51 + rank, n_out=4, n_slash=3)
    iv, is_ = random_selection(B, Hq, N, 24, 40, 52 + rank)
    q, k, v, do = (dev_bf16(x[n]) for n in ("q", "k", "v", "dout"))
    q_r = vs.ring_permute(q, W, "zigzag", only_rank=rank)
    do_r = vs.ring_permute(do, W, "zigzag", only_rank=rank)
    ksh, vsh = vs.ring_permute(k, W, "zigzag"), vs.ring_permute(v, W, "zigzag")
    wk = vs.ZigZagWorker(B, N, Hq, Hkv, d, iv.shape[-1], is_.shape[-1], W, rank=rank)
    wk.v_idx.copy_(torch.from_numpy(iv))
    wk.s_idx.copy_(torch.from_numpy(is_))
    wk.build_index(q_r, ksh)
    o, lse = wk.forward(q_r, ksh, vsh)
    dq, dk, dv = wk.backward(do_r)
    torch.cuda.synchronize()
    wk.check()
    pos = oracle.ring_positions(N, W, rank, "zigzag")
    lse_all = torch.cat(lse, dim=2).cpu().numpy().astype(np.float64)  # [B, Hq, 2C] in local order
    for b in range(B):
        p = oracle.Problem(host_f64(x["q"])[b:b + 1, pos], host_f64(x["k"])[b:b + 1], host_f64(x["v"])[b:b + 1],
                           iv[b:b + 1], is_[b:b + 1], 1 / math.sqrt(d), dout=host_f64(x["dout"])[b:b + 1, pos],
                           qpos=pos, n_global=N)
        rows = np.array([(0, h, i) for h in range(Hq) for i in range(len(pos))], np.int32)
        o_ref, lse_ref, dq_ref = oracle.rows(p, rows)
        o_g = host_f64(o)[b]
        dq_g = host_f64(dq)[b]
        assert rel_l2(np.stack([o_g[i, h] for h in range(Hq) for i in range(len(pos))]), o_ref) <= TOL
        assert rel_l2(np.stack([dq_g[i, h] for h in range(Hq) for i in range(len(pos))]), dq_ref) <= TOL
        got_lse = np.concatenate([lse_all[b, h] for h in range(Hq)])
        fin = np.isfinite(lse_ref)
        np.testing.assert_array_equal(np.isfinite(got_lse), fin)
        assert np.max(np.abs(got_lse[fin] - lse_ref[fin]), initial=0.0) <= 1e-3
        # each source shard's dK / dV: the contribution of this worker's rows
        for src in range(W):
            kpos = oracle.ring_positions(N, W, src, "zigzag")
            keys = np.array([(0, 0, m) for m in kpos], np.int32)
            dk_ref, dv_ref = oracle.keys(p, keys)
            assert rel_l2(host_f64(dk[src])[b, :, 0], dk_ref) <= TOL, (b, src)
            assert rel_l2(host_f64(dv[src])[b, :, 0], dv_ref) <= TOL, (b, src)
