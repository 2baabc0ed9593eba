"""Ring-layout work counts on the GPU (MTraining sections 2, 3.3, 4.2:
Striped vs ZigZag Ring Attention) against the oracle, through the C ABI:
integer counts, so equality is exact."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from vs_testutil import random_selection

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ring_work_n256_w2.json")


@pytest.fixture(scope="module")
def vs():
    import dynamic_vertical_slash_gb300 as m

    m.lib()
    return m


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def _run(vs, iv, is_, N, W, layout):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    out = vs.vs_ring_work(_dev(iv), _dev(is_), N, W, layout, ws=ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), vs.vs_check_status(ws)


def _area(iv, is_, N):
    """Mask entries from the lists in closed form: columns, offsets, minus
    the entries that are on both."""
    tot = 0
    for b in range(iv.shape[0]):
        for h in range(iv.shape[1]):
            m = iv[b, h][iv[b, h] >= 0].astype(np.int64)
            o = np.sort(is_[b, h][is_[b, h] >= 0].astype(np.int64))
            tot += int((N - m).sum() + (N - o).sum() - np.searchsorted(o, N - m, side="left").sum())
    return tot


def test_hand_worked_example(vs):
    g = json.load(open(GOLDEN))
    N = g["N"]
    iv = np.zeros((1, 1, 1), np.int32)
    is_ = np.arange(N, dtype=np.int32).reshape(1, 1, N)
    for layout in ("striped", "zigzag"):
        got, st = _run(vs, iv, is_, N, g["W"], layout)
        assert st == 0 and got.tolist() == g[layout], layout


@pytest.mark.parametrize("layout", ["striped", "zigzag"])
@pytest.mark.parametrize("N,W,kv,ks,seed", [(1024, 4, 17, 40, 1), (2048, 8, 64, 200, 2), (768, 3, 5, 300, 3),
                                            (1024, 1, 30, 30, 4)])
def test_matches_oracle(vs, layout, N, W, kv, ks, seed):
    iv, is_ = random_selection(2, 3, N, kv, ks, seed)
    # pad some heads with -1 (top-p lists)
    iv = np.concatenate([iv, np.full((2, 3, 3), -1, np.int32)], -1)
    is_[1, 2, ks // 2:] = -1
    got, st = _run(vs, iv, is_, N, W, layout)
    assert st == 0
    np.testing.assert_array_equal(got, oracle.ring_work(iv, is_, N, W, layout))


def test_full_size_selection_totals(vs):
    # 512K tokens, 8 workers, 16 heads of kv = 1024 / ks = 2048 random lists:
    # the counts sum to the mask area in closed form for both layouts
    N, W = 524288, 8
    iv, is_ = random_selection(1, 16, N, 1024, 2048, 9)
    area = _area(iv, is_, N)
    for layout in ("striped", "zigzag"):
        got, st = _run(vs, iv, is_, N, W, layout)
        assert st == 0 and int(got.sum()) == area, layout


def test_zigzag_balances_full_causal(vs):
    N, W = 65536, 8
    iv = np.zeros((1, 1, 1), np.int32)
    is_ = np.arange(N, dtype=np.int32).reshape(1, 1, N)
    got, st = _run(vs, iv, is_, N, W, "zigzag")
    tot = got.sum(1)
    assert st == 0 and (tot == tot[0]).all() and int(tot.sum()) == N * (N + 1) // 2


def test_bad_lists(vs):
    iv = np.array([[[5, 3]]], np.int32)
    is_ = np.array([[[1]]], np.int32)
    _, st = _run(vs, iv, is_, 256, 2, "striped")
    assert st == 4
    with pytest.raises(vs.VSError):
        vs.vs_ring_work(_dev(iv), _dev(is_), 250, 2, "striped")
