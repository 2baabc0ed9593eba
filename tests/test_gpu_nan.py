"""Non-finite inputs: every call returns with a clean status (no wait runs
out: the kernels' loops have fixed trip counts, and the forward's per-pair
re-basing runs at most once per pair), and a NaN in one query row n of head h
stays where the computation puts it.  The forward takes a row whose softmax
sum is not a positive number (here NaN) for an empty row: O = 0, LSE = -inf.

By the definitions, O, LSE and dQ of row n, and dK, dV of the keys in row
n's mask depend on that row.  The kernels keep O, LSE, dQ and dV to exactly
that (P of a masked entry is a selected zero, and the other operands are
finite); dK is a tile-level product, dK += dS^T Q over a unit's 64 rows, in
which the NaN of Q's row n (and dS = 0 * (dP - D_n) with D_n = NaN) reaches
every key of the units that contain row n.  So dK is checked on the keys
that no unit containing row n touches: keys of later key tiles that no head
selected as a column.  Everything checked must match the oracle run on the
same inputs without the NaN.  A NaN in the estimator's observation window
reaches the scores; the selection it returns is still a valid list (sorted,
unique, in range) and the index accepts it."""
import ctypes
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


@pytest.mark.parametrize("d", [64, 128])
def test_nan_query_row_stays_in_its_outputs(vs, d):
    B, N, Hq, Hkv, kv, ks = 1, 1088, 4, 2, 24, 40
    w, x = make_inputs(B, N, Hq, Hkv, d, seed=61 + d, n_out=3, n_slash=2)
    iv, is_ = random_selection(B, Hq, N, kv, ks, 62 + d)
    n0, h0 = 700, 1  # a row in the middle of a query tile
    q = dev_bf16(x["q"])
    q[0, n0, h0, 5] = float("nan")
    k, v, do = dev_bf16(x["k"]), dev_bf16(x["v"]), dev_bf16(x["dout"])
    arena = vs.vs_build_block_index(q, k, torch.from_numpy(iv).cuda(), torch.from_numpy(is_).cuda())
    o, lse = vs.vs_attn_fwd(q, k, v, arena)
    dq, dk, dv = vs.vs_attn_bwd(q, k, v, o, lse, do, arena, kv)
    torch.cuda.synchronize()
    assert vs.vs_check_status(arena) == 0

    p = oracle.Problem(host_f64(x["q"]), host_f64(x["k"]), host_f64(x["v"]), iv, is_, 1 / math.sqrt(d),
                       dout=host_f64(x["dout"]))
    ref = oracle.attention(p)
    row_mask = oracle.mask_dense(p, 0, h0)[n0]  # the keys row n0 attends
    assert row_mask.any()
    # the poisoned row itself: the forward takes a row whose softmax sum is
    # not a positive number for an empty row (O = 0, LSE = -inf)
    assert float(o[0, n0, h0].abs().max()) == 0.0 and float(lse[0, h0, n0]) == float("-inf")
    # every other row: O, LSE, dQ as without the NaN
    keep = np.ones((B, N, Hq), bool)
    keep[0, n0, h0] = False
    O, DQ = host_f64(o), host_f64(dq)
    assert np.isfinite(O[keep]).all() and np.isfinite(DQ[keep]).all()
    assert rel_l2(O[keep], ref["o"][keep]) <= TOL
    assert rel_l2(DQ[keep], ref["dq"][keep]) <= TOL
    L = lse.cpu().numpy().astype(np.float64).transpose(0, 2, 1)  # [B, N, Hq]
    Lr = ref["lse"].transpose(0, 2, 1)
    fin = np.isfinite(Lr[keep])
    np.testing.assert_array_equal(np.isfinite(L[keep]), fin)
    assert np.max(np.abs(L[keep][fin] - Lr[keep][fin]), initial=0.0) <= 1e-3
    # dV: keys outside the row's mask (of its KV head), and every key of the
    # other KV heads
    g = Hq // Hkv
    hk0 = h0 // g
    vkeep = np.ones((B, N, Hkv), bool)
    vkeep[0, row_mask, hk0] = False
    DK, DV = host_f64(dk), host_f64(dv)
    assert np.isfinite(DV[vkeep]).all()
    assert rel_l2(DV[vkeep], ref["dv"][vkeep]) <= TOL
    # dK: the other KV heads, and the keys of KV head hk0 in key tiles that
    # start after row n0 and that no head of the group selected as a column
    kkeep = np.ones((B, N, Hkv), bool)
    kkeep[0, :, hk0] = False
    later = np.arange(N) >= 128 * (n0 // 128 + 1)
    later[np.unique(iv[0, hk0 * g:(hk0 + 1) * g])] = False
    kkeep[0, later, hk0] = True
    assert later.sum() > 100
    assert np.isfinite(DK[kkeep]).all()
    assert rel_l2(DK[kkeep], ref["dk"][kkeep]) <= TOL


def test_nan_in_the_observation_window_gives_a_valid_selection(vs):
    B, N, Hq, Hkv, d, kv, ks = 1, 1024, 2, 1, 64, 32, 32
    w, x = make_inputs(B, N, Hq, Hkv, d, seed=63, n_out=4)
    q, k = dev_bf16(x["q"]), dev_bf16(x["k"])
    q[0, N - 10, 0, 3] = float("nan")  # one of head 0's last 64 rows
    sh = vs.make_shape(q, k)
    ws = torch.zeros(vs.lib().vs_estimate_workspace(ctypes.byref(sh), 64), dtype=torch.uint8, device="cuda")
    iv, is_ = vs.vs_estimate(q, k, kv, ks, d ** -0.5, 64, ws=ws)
    torch.cuda.synchronize()
    assert vs.vs_check_status(ws) == 0
    for lists, n in ((iv, kv), (is_, ks)):
        a = lists.cpu().numpy()
        assert a.shape == (B, Hq, n)
        assert ((a >= 0) & (a < N)).all()
        assert (np.diff(a, axis=-1) > 0).all()  # sorted and unique
    # head 1 is untouched: its selection equals the one without the NaN
    iv_c, is_c = vs.vs_estimate(dev_bf16(x["q"]), k, kv, ks, d ** -0.5, 64)
    assert torch.equal(iv[0, 1], iv_c[0, 1]) and torch.equal(is_[0, 1], is_c[0, 1])
    # the index accepts the lists and the attention runs
    arena = vs.vs_build_block_index(q, k, iv, is_)
    vs.vs_attn_fwd(q, k, dev_bf16(x["v"]), arena)
    torch.cuda.synchronize()
    assert vs.vs_check_status(arena) == 0
