"""The striped ring driver (one worker's ring steps on one GPU) in both step
orders: the flat ring (src = rank - s mod W) and the hierarchical order of
Hierarchical Balanced Sparse Ring Attention (inner rings of `inner` cards
inside an outer ring of nodes).  The order changes only the summation order:
merged O / LSE, accumulated dQ and each source shard's dK / dV agree between
the orders and with the fp64 oracle's global computation on the worker's
rows."""
import math

import numpy as np
import pytest
import torch

import oracle
from vs_testutil import dev_bf16, host_f64, make_inputs, random_selection, rel_l2

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _run(vs, x, iv, is_, W, rank, inner, N, Hq, Hkv, d):
    q, k, v, do = (dev_bf16(x[n]) for n in ("q", "k", "v", "dout"))
    q_r = vs.striped_permute(q, W, only_rank=rank)
    do_r = vs.striped_permute(do, W, only_rank=rank)
    ksh, vsh = vs.striped_permute(k, W), vs.striped_permute(v, W)
    wk = vs.StripedWorker(1, N, Hq, Hkv, d, iv.shape[-1], is_.shape[-1], W, rank=rank, inner=inner)
    wk.v_idx.copy_(torch.from_numpy(iv))
    wk.s_idx.copy_(torch.from_numpy(is_))
    wk.build_index(q_r, ksh)
    o, lse = wk.forward(q_r, ksh, vsh)
    dq, dk, dv = wk.backward(do_r)
    torch.cuda.synchronize()
    wk.check()
    return {"o": host_f64(o), "lse": lse.cpu().numpy().astype(np.float64), "dq": host_f64(dq), "dk": host_f64(dk),
            "dv": host_f64(dv), "src": [wk.source(s) for s in range(W)]}


@pytest.mark.parametrize("rank", [0, 2])
def test_hierarchical_order_matches_flat_and_oracle(rank):
    import dynamic_vertical_slash_gb300 as vs

    B, N, Hq, Hkv, d, W, inner = 1, 2048, 2, 1, 64, 4, 2
    w, x = make_inputs(B, N, Hq, Hkv, d, seed=41, n_out=4, n_slash=3)
    iv, is_ = random_selection(B, Hq, N, 24, 40, 42)
    flat = _run(vs, x, iv, is_, W, rank, 0, N, Hq, Hkv, d)
    hier = _run(vs, x, iv, is_, W, rank, inner, N, Hq, Hkv, d)
    assert sorted(hier["src"]) == list(range(W)) and hier["src"] != flat["src"]
    for key in ("o", "dq", "dk", "dv"):
        assert rel_l2(hier[key], flat[key]) <= 2e-3, key
    fin = np.isfinite(flat["lse"])
    np.testing.assert_array_equal(np.isfinite(hier["lse"]), fin)
    assert np.max(np.abs(hier["lse"][fin] - flat["lse"][fin]), initial=0.0) <= 1e-4
    # against the global computation on the worker's rows
    pos = oracle.stripe_positions(N, W, 64, rank)
    p = oracle.Problem(host_f64(x["q"])[:, pos], host_f64(x["k"]), host_f64(x["v"]), iv, is_, 1 / math.sqrt(d),
                       dout=host_f64(x["dout"])[:, pos], qpos=pos, n_global=N)
    rows = np.array([(0, h, i) for h in range(Hq) for i in range(len(pos))], np.int32)
    o_ref, lse_ref, dq_ref = oracle.rows(p, rows)
    o_h = np.stack([hier["o"][0, i, h] for h in range(Hq) for i in range(len(pos))])
    dq_h = np.stack([hier["dq"][0, i, h] for h in range(Hq) for i in range(len(pos))])
    assert rel_l2(o_h, o_ref) <= TOL
    assert rel_l2(dq_h, dq_ref) <= TOL
    for src in range(W):
        kpos = oracle.stripe_positions(N, W, 64, src)
        keys = np.array([(0, 0, m) for m in kpos], np.int32)
        dk_ref, dv_ref = oracle.keys(p, keys)
        assert rel_l2(hier["dk"][src, 0, :, 0], dk_ref) <= TOL, src
        assert rel_l2(hier["dv"][src, 0, :, 0], dv_ref) <= TOL, src
