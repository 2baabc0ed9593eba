"""Per-KV-group shared selection on the GPU (vs_estimate_group) against the
oracle: replay on the GPU's own fp32 scores (group sums in fp32, head
order, as the kernel adds them), planted columns, and the layer option."""
import math

import numpy as np
import pytest
import torch

import oracle
from vs_testutil import dev_bf16, host_f64, make_inputs, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vs():
    import dynamic_vertical_slash_gb300 as m

    m.lib()
    return m


@pytest.mark.parametrize("B,N,Hq,Hkv,d,kv,ks,seed", [(1, 2048, 4, 2, 64, 40, 64, 1), (2, 1024, 8, 1, 128, 33, 17, 2)])
def test_group_replay(vs, B, N, Hq, Hkv, d, kv, ks, seed):
    w, x = make_inputs(B, N, Hq, Hkv, d, seed, n_out=5, n_slash=4)
    q, k = dev_bf16(x["q"]), dev_bf16(x["k"])
    vsc = torch.empty(B, Hq, N, device="cuda")
    ssc = torch.empty(B, Hq, N, device="cuda")
    iv, is_ = vs.vs_estimate(q, k, kv, ks, w.scale, v_score=vsc, s_score=ssc, shared=True)
    torch.cuda.synchronize()
    g = Hq // Hkv
    ref = oracle.select_group(vsc.cpu().numpy(), ssc.cpu().numpy(), kv, ks, g, dtype=np.float32)
    np.testing.assert_array_equal(iv.cpu().numpy(), ref[0])
    np.testing.assert_array_equal(is_.cpu().numpy(), ref[1])
    # per-head scores are the estimator's
    vsc2, ssc2 = torch.empty_like(vsc), torch.empty_like(ssc)
    vs.vs_estimate(q, k, kv, ks, w.scale, v_score=vsc2, s_score=ssc2)
    assert torch.equal(vsc, vsc2) and torch.equal(ssc, ssc2)


def test_group_planted_columns(vs):
    w, x = make_inputs(1, 2048, 4, 2, 64, seed=21, n_out=6, n_slash=5)
    q, k = dev_bf16(x["q"]), dev_bf16(x["k"])
    iv, _ = vs.vs_estimate(q, k, 6, 5, w.scale, shared=True)
    ivh = iv.cpu().numpy()
    for h in range(4):
        np.testing.assert_array_equal(ivh[0, h], np.sort(x["planted_cols"][0][h // 2]))
    v_ref, s_ref = oracle.estimate(host_f64(x["q"]), host_f64(x["k"]), 64, w.scale)
    np.testing.assert_array_equal(ivh, oracle.select_group(v_ref, s_ref, 6, 5, 2)[0])


def test_layer_shared_option(vs):
    w, x = make_inputs(1, 1024, 4, 2, 64, seed=31, n_out=4, n_slash=3)
    q, k, v = dev_bf16(x["q"]), dev_bf16(x["k"]), dev_bf16(x["v"])
    layer = vs.VSAttention(1, 1024, 4, 2, 64, 24, 40, shared=True)
    layer.forward(q, k, v)
    torch.cuda.synchronize()
    layer.check()
    ivh = layer.v_idx.cpu().numpy()
    assert np.array_equal(ivh[0, 0], ivh[0, 1]) and np.array_equal(ivh[0, 2], ivh[0, 3])
    # attention on the oracle's own group selection matches the oracle
    v_ref, s_ref = oracle.estimate(host_f64(x["q"]), host_f64(x["k"]), 64, w.scale)
    ivr, isr = oracle.select_group(v_ref, s_ref, 24, 40, 2)
    o, lse = layer.forward(q, k, v, selection=(torch.from_numpy(ivr).cuda(), torch.from_numpy(isr).cuda()))
    dq, dk, dv = layer.backward(dev_bf16(x["dout"]))
    torch.cuda.synchronize()
    ref = oracle.attention(oracle.Problem(host_f64(x["q"]), host_f64(x["k"]), host_f64(x["v"]), ivr, isr,
                                          1 / math.sqrt(64), dout=host_f64(x["dout"])))
    for name, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert rel_l2(host_f64(t), ref[name]) <= 1e-2, name
