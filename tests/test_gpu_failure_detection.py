"""Failure detection on the GPU without a fault: a bounded device wait that
nothing satisfies runs out, the kernel records VS_ERR_TIMEOUT in the caller's
status word and returns, the CTA's other waiting warp leaves on the abort
flag, and the CUDA context keeps working (a small attention call afterwards
still matches the oracle)."""
import math
import time

import numpy as np
import pytest
import torch

import oracle
from vs_testutil import dev_bf16, host_f64, make_inputs, random_selection, rel_l2

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_context_survives():
    import dynamic_vertical_slash_gb300 as vs

    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    vs.vs_selftest_wait_timeout(ws)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    words = ws[:8].cpu().numpy().view(np.int32)
    assert words[1] == 2, "both warps must return after giving up (got %d)" % words[1]
    assert vs.vs_check_status(ws) == 5  # VS_ERR_TIMEOUT
    assert vs.status_string(5).startswith("VS_ERR_TIMEOUT")
    assert vs.vs_check_status(ws) == 0  # reading resets the word
    assert 1.0 <= elapsed <= 30.0, elapsed

    # the context is still usable: a small sparse attention matches the oracle
    B, N, Hq, Hkv, d = 1, 512, 2, 1, 64
    w, x = make_inputs(B, N, Hq, Hkv, d, seed=31, n_out=2, n_slash=1)
    iv, is_ = random_selection(B, Hq, N, 8, 16, 32)
    q, k, v = dev_bf16(x["q"]), dev_bf16(x["k"]), dev_bf16(x["v"])
    arena = vs.vs_build_block_index(q, k, torch.from_numpy(iv).cuda(), torch.from_numpy(is_).cuda())
    o, lse = vs.vs_attn_fwd(q, k, v, arena)
    torch.cuda.synchronize()
    assert vs.vs_check_status(arena) == 0
    p = oracle.Problem(host_f64(x["q"]), host_f64(x["k"]), host_f64(x["v"]), iv, is_, 1 / math.sqrt(d))
    ref = oracle.attention(p)
    assert rel_l2(host_f64(o), ref["o"]) <= 1e-2


def test_estimator_skips_its_work_after_a_recorded_failure():
    # a failure already in the status word (as a timed-out kernel of the same
    # call would leave it) makes every estimator kernel skip: no kernel reads
    # scratch that a failed kernel left unwritten, the outputs stay as they
    # were, and the code is reported once
    import dynamic_vertical_slash_gb300 as vs

    B, N, Hq, Hkv, d = 1, 1024, 2, 1, 64
    w, x = make_inputs(B, N, Hq, Hkv, d, seed=32, n_out=4, n_slash=1)
    q, k = dev_bf16(x["q"]), dev_bf16(x["k"])
    iv_ok, is_ok = vs.vs_estimate(q, k, 16, 16)
    import ctypes

    need = vs.lib().vs_estimate_workspace(ctypes.byref(vs.make_shape(q, k)), 64)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ws[:4].view(torch.int32).fill_(5)  # VS_ERR_TIMEOUT
    iv = torch.full((B, Hq, 16), -7, dtype=torch.int32, device="cuda")
    is_ = torch.full((B, Hq, 16), -7, dtype=torch.int32, device="cuda")
    vsc = torch.full((B, Hq, N), -1.0, device="cuda")
    ssc = torch.full((B, Hq, N), -1.0, device="cuda")
    vs.vs_estimate(q, k, 16, 16, v_idx=iv, s_idx=is_, v_score=vsc, s_score=ssc, ws=ws)
    torch.cuda.synchronize()
    assert bool((iv == -7).all()) and bool((is_ == -7).all())
    assert bool((vsc == -1).all()) and bool((ssc == -1).all())
    assert vs.vs_check_status(ws) == 5
    # with the word read (and reset) the same workspace computes again
    vs.vs_estimate(q, k, 16, 16, v_idx=iv, s_idx=is_, v_score=vsc, s_score=ssc, ws=ws)
    torch.cuda.synchronize()
    assert vs.vs_check_status(ws) == 0
    assert torch.equal(iv, iv_ok) and torch.equal(is_, is_ok)
